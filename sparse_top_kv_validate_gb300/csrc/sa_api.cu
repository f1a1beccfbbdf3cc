// sa_api.cu -- the library's C ABI: host-side argument checks, work planning
// (units, splits, workspace carving) and kernel launches.  Nothing here
// allocates, frees or synchronises; everything is enqueued on the caller's
// stream.
#include <cuda_runtime.h>
#include <atomic>
#include <cmath>
#include <mutex>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/sa.h"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t dtype_bytes(int dt) {
  switch (dt) {
    case SA_F32: return 4;
    case SA_F16: return 2;
    case SA_BF16: return 2;
    default: return 0;
  }
}

// Half-open byte ranges [a, a+na) and [b, b+nb) intersect.
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

struct DeviceShape {
  int sms = 152;
};

DeviceShape device_shape() {
  DeviceShape d;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      d.sms = n;
  }
  return d;
}

void plan_simt_splits(int64_t n_cand, int64_t* chunk_out, int64_t* splits_out) {
  int64_t splits = (n_cand + 255) / 256;
  if (splits < 1) splits = 1;
  if (splits > 64) splits = 64;
  int64_t chunk = (n_cand + splits - 1) / splits;
  if (chunk < 1) chunk = 1;
  *chunk_out = chunk;
  *splits_out = (n_cand + chunk - 1) / chunk > 0 ? (n_cand + chunk - 1) / chunk : 1;
}

// A gather request after planning: which kernel runs, its grid, and where
// its scratch lives inside the caller's workspace (nothing in it needs to be
// initialised: every word is written before it is read).
struct Plan {
  sa::GatherArgs g;
  bool stream = false;
  bool fp8 = false;
  bool fp8_tc = false;       // the tcgen05 kernels (128-key tiles)
  bool fp8_combine = false;  // FP8 key splits merged by launch_combine
  int grid = 0;
  size_t off_pos = 0, off_meta = 0, off_part_o = 0, off_part_ml = 0, off_kdec = 0, bytes = 0;
};

int stream_grid() {
  const int sms = device_shape().sms;
  // one CTA per SM: the kernel's shared-memory rings fill the SM
  return sms > 0 ? sms : 152;
}

// Fill the unit geometry, pick the kernel and lay out the workspace for a
// request whose source, shape and tensor fields are set.
int plan_gather(Plan& pl, int dtype) {
  sa::GatherArgs& g = pl.g;
  g.g = g.Hq / g.Hkv;
  if (g.source == sa::kSparse && g.I == g.Hq && g.g > 1) {
    g.n_groups = g.Hq;  // each query head has its own index row
    g.hpu = 1;
  } else {
    g.n_groups = g.Hkv;
    g.hpu = g.g;
  }
  g.units = g.B * g.n_groups * g.Sq;
  pl.stream = sa::gather_uses_mma(g, dtype) &&
              (g.source != sa::kPaged || (g.B <= sa::stream_max_batch_paged() &&
                                          g.max_pages * g.page_tokens < (int64_t(1) << 31)));
  const int64_t irows = g.B * g.I * g.Sq;
  if (pl.stream) {
    pl.grid = stream_grid();
    const int64_t gw = static_cast<int64_t>(pl.grid) * sa::stream_warps(static_cast<int>(g.D));
    g.tiles_per_unit = (g.n_cand + 15) / 16;
    g.n_cand_pad = g.tiles_per_unit * 16;
    if (g.units * g.tiles_per_unit >= (int64_t(1) << 31) ||
        g.B * g.Hkv * ((g.max_pages * g.page_tokens + 15) / 16) >= (int64_t(1) << 31) ||
        irows * g.n_cand_pad >= (int64_t(1) << 40))
      return SA_ERR_UNSUPPORTED;
    if (g.source != sa::kPaged) {
      const int64_t nt = g.units * g.tiles_per_unit;
      g.tiles_per_warp = (nt + gw - 1) / gw;
      if (g.tiles_per_warp < 1) g.tiles_per_warp = 1;
    }
    size_t off = 0;
    if (g.source == sa::kSparse) {
      pl.off_pos = off;
      off += align_up(static_cast<size_t>(irows * g.n_cand_pad) * sizeof(int32_t));
    }
    pl.off_meta = off;
    off += align_up(sizeof(int64_t) + static_cast<size_t>(g.B + 1) * sizeof(int32_t));
    const size_t parts = static_cast<size_t>(gw) * 2 * g.hpu;
    pl.off_part_o = off;
    off += align_up(parts * g.D * sizeof(float));
    pl.off_part_ml = off;
    off += align_up(parts * 2 * sizeof(float));
    pl.bytes = off;
  } else {
    if ((g.D + 31) / 32 > 16) return SA_ERR_UNSUPPORTED;
    plan_simt_splits(g.n_cand, &g.chunk, &g.splits);
    if (g.splits > 1) {
      const size_t parts = static_cast<size_t>(g.units * g.splits * g.hpu);
      pl.off_part_o = 0;
      pl.off_part_ml = align_up(parts * g.Dv * sizeof(float));
      pl.bytes = pl.off_part_ml + align_up(parts * 2 * sizeof(float));
    }
  }
  return SA_OK;
}

// FP8 hybrid-record decode: planned positions (as the stream path), then the
// tcgen05 kernel (128-head blocks, 128-key tiles, three CTAs per output block)
// or the warp-level MMA kernel (32-head blocks, 16-key tiles); key splits are
// merged by the combine kernel.
int plan_fp8(Plan& pl) {
  sa::GatherArgs& g = pl.g;
  pl.fp8 = true;
  g.g = g.Hq / g.Hkv;
  g.n_groups = g.Hkv;  // 1: every query head shares the latent head
  g.hpu = g.g;
  g.units = g.B * g.n_groups * g.Sq;
  pl.fp8_tc = sa::fp8_tc_supported(g);
  const int64_t sms = device_shape().sms > 0 ? device_shape().sms : 152;
  if (pl.fp8_tc) {
    // 128-key tiles; (unit, 128-head block, split) x 3 dim parts, one CTA per SM
    g.tiles_per_unit = (g.n_cand + 127) / 128;
    g.n_cand_pad = g.tiles_per_unit * 128;
    const int64_t blocks = g.units * (g.Hq / 128) * 3;
    int64_t splits = sms / (blocks > 0 ? blocks : 1);
    const int64_t min_splits = (g.tiles_per_unit + sa::fp8_tc_max_tiles() - 1) / sa::fp8_tc_max_tiles();
    if (splits < min_splits) splits = min_splits;
    if (splits < 1) splits = 1;
    if (splits > g.tiles_per_unit) splits = g.tiles_per_unit;
    g.chunk = (g.tiles_per_unit + splits - 1) / splits;
    g.splits = (g.tiles_per_unit + g.chunk - 1) / g.chunk;
    if (g.units * (g.Hq / 128) * g.splits * 3 >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  } else {
    g.tiles_per_unit = (g.n_cand + 15) / 16;
    g.n_cand_pad = g.tiles_per_unit * 16;
    const int64_t blocks = g.units * (g.Hq / 32);
    const int64_t slots = sms * 2;  // 2 CTAs per SM
    int64_t splits = slots / (blocks > 0 ? blocks : 1);
    const int64_t min_splits = (g.tiles_per_unit + sa::fp8_chunk_tiles_max() - 1) /
                               sa::fp8_chunk_tiles_max();
    if (splits < min_splits) splits = min_splits;
    if (splits < 1) splits = 1;
    if (splits > g.tiles_per_unit) splits = g.tiles_per_unit > 0 ? g.tiles_per_unit : 1;
    g.chunk = (g.tiles_per_unit + splits - 1) / splits;  // tiles per chunk
    g.splits = (g.tiles_per_unit + g.chunk - 1) / g.chunk;
  }
  if (g.splits < 1) g.splits = 1;
  const int64_t irows = g.B * g.I * g.Sq;
  size_t off = 0;
  pl.off_pos = off;
  off += align_up(static_cast<size_t>(irows * g.n_cand_pad) * sizeof(int32_t));
  pl.fp8_combine = g.splits > 1 && !(pl.fp8_tc && sa::fp8_tc_cluster_merge(g.splits, g.units * (g.Hq / 128) * 3));
  if (pl.fp8_combine) {
    const size_t parts = static_cast<size_t>(g.units * g.splits * g.hpu);
    pl.off_part_o = off;
    off += align_up(parts * g.Dv * sizeof(float));
    pl.off_part_ml = off;
    off += align_up(parts * 2 * sizeof(float));
  }
  if (pl.fp8_tc) {
    pl.off_kdec = off;
    off += align_up(static_cast<size_t>(g.units * g.n_cand_pad) * sa::fp8_tc_decoded_row_bytes());
  }
  pl.bytes = off;
  return SA_OK;
}

int check_workspace(const Plan& pl, void* ws, size_t ws_bytes) {
  if (pl.bytes == 0) return SA_OK;
  if (!ws || ws_bytes < pl.bytes) return SA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return SA_ERR_ALIGN;
  return SA_OK;
}

// Carve the workspace; for the stream path return the planned-position area.
void carve(Plan& pl, void* ws) {
  sa::GatherArgs& g = pl.g;
  char* base = static_cast<char*>(ws);
  if (pl.bytes == 0) return;
  if (pl.fp8) {
    g.pos = reinterpret_cast<const int32_t*>(base + pl.off_pos);
    if (pl.fp8_combine) {
      g.part_o = reinterpret_cast<float*>(base + pl.off_part_o);
      g.part_ml = reinterpret_cast<float*>(base + pl.off_part_ml);
    }
    if (pl.fp8_tc) g.fp8_kdec = base + pl.off_kdec;
    return;
  }
  g.part_o = reinterpret_cast<float*>(base + pl.off_part_o);
  g.part_ml = reinterpret_cast<float*>(base + pl.off_part_ml);
  if (pl.stream) {
    g.meta = reinterpret_cast<int64_t*>(base + pl.off_meta);
    g.pref_out = reinterpret_cast<int32_t*>(base + pl.off_meta + sizeof(int64_t));
    if (g.source == sa::kSparse) g.pos = reinterpret_cast<const int32_t*>(base + pl.off_pos);
  }
}

// Measurement hook: events recorded around the dominant kernel of each call
// made from this host thread (sa_set_kernel_events).
thread_local void* t_ev_before = nullptr;
thread_local void* t_ev_after = nullptr;

int run_plan(Plan& pl, int dtype, cudaStream_t st) {
  sa::GatherArgs& g = pl.g;
  g.ev_before = t_ev_before;
  g.ev_after = t_ev_after;
  if (pl.fp8) {
    if (pl.fp8_tc) {
      if (sa::launch_fp8_tc(g, st) != 0) return SA_ERR_LAUNCH;  // brackets its attention kernel
    } else {
      sa::mark_event(g.ev_before, st);
      const int rc = sa::launch_fp8_decode(g, st);
      sa::mark_event(g.ev_after, st);
      if (rc != 0) return SA_ERR_LAUNCH;
    }
    if (pl.fp8_combine && sa::launch_combine(g, SA_BF16, st) != 0) return SA_ERR_LAUNCH;
    return SA_OK;
  }
  if (pl.stream) {
    sa::mark_event(g.ev_before, st);
    const int rc = sa::launch_gather_stream(g, dtype, pl.grid, st);
    sa::mark_event(g.ev_after, st);
    if (rc != 0) return SA_ERR_LAUNCH;
    if (sa::launch_stream_combine(g, dtype, st) != 0) return SA_ERR_LAUNCH;
    return SA_OK;
  }
  sa::mark_event(g.ev_before, st);
  const int rc = sa::launch_gather_simt(g, dtype, st);
  sa::mark_event(g.ev_after, st);
  if (rc != 0) return SA_ERR_LAUNCH;
  if (sa::launch_combine(g, dtype, st) != 0) return SA_ERR_LAUNCH;
  return SA_OK;
}

// ---- sparse decode: checks + plan ----------------------------------------------

// [IS] validate_bias_shape: rank <= 4, each axis 1 or the extent of the axis
// of [B, Hq, Sq, T] it lines up with from the right.  On success the element
// strides of the four logical axes (0 on broadcast axes) go to st.
bool bias_strides(const sa_sparse_params* p, int64_t st[4]) {
  const int64_t target[4] = {p->B, p->Hq, p->Sq, p->T};
  if (p->bias_rank < 0 || p->bias_rank > 4) return false;
  const int r = static_cast<int>(p->bias_rank);
  int64_t run = 1;
  for (int ax = 3; ax >= 0; --ax) {
    const int k = ax - (4 - r);  // index into bias_dims, < 0 for a missing leading axis
    if (k < 0) {
      st[ax] = 0;
      continue;
    }
    const int64_t e = p->bias_dims[k];
    if (e != 1 && e != target[ax]) return false;
    st[ax] = (e == 1) ? 0 : run;
    run *= e;
  }
  return true;
}

// `query` = 1 for a workspace-size query, which needs no output pointer.
int check_sparse(const sa_sparse_params* p, int query = 0) {
  if (!p || !p->q || !p->k_cache || (!p->y && !query)) return SA_ERR_NULL;
  if (p->reserved_ != 0 || (p->options & ~(SA_OPT_ROW_COPIES | SA_OPT_FP8_WARP_MMA)))
    return SA_ERR_UNSUPPORTED;
  if (p->bias) {
    int64_t st[4];
    if (!bias_strides(p, st)) return SA_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(p->bias) % 4) return SA_ERR_ALIGN;
  }
  if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Sq <= 0 || p->D <= 0 || p->T <= 0)
    return SA_ERR_SHAPE;
  if (p->Hq % p->Hkv != 0) return SA_ERR_SHAPE;
  if (!(p->I == 1 || p->I == p->Hkv || p->I == p->Hq)) return SA_ERR_SHAPE;
  if (p->K < 0 || p->window < 0 || p->past_len < 0) return SA_ERR_SHAPE;
  if (p->K == 0 && p->window == 0) return SA_ERR_SHAPE;
  if (p->K > 0 && !p->idx) return SA_ERR_NULL;
  if (!std::isfinite(p->scale) || !std::isfinite(p->softcap) || p->softcap < 0.f)
    return SA_ERR_SHAPE;
  if (p->kv_dtype == SA_FP8_E4M3_B64) {
    // hybrid records: bf16 Q/Y, one latent head, 512 E4M3 dims + 64 bf16 dims
    if (p->q_dtype != SA_BF16) return SA_ERR_DTYPE;
    if (p->D != 576 || p->n_rope != 64 || p->Dv != p->D || p->Hkv != 1 || p->I != 1 ||
        p->Hq % 32 != 0 || p->k_cur)
      return SA_ERR_UNSUPPORTED;
    if (p->record_stride < 648 || p->record_stride % 8 != 0) return SA_ERR_SHAPE;
    if (p->B * p->T >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(p->k_cache) % 8 || !aligned16(p->q) || !aligned16(p->y ? p->y : p->q))
      return SA_ERR_ALIGN;
    const size_t qbytes = static_cast<size_t>(p->B * p->Hq * p->Sq * p->D) * 2;
    const size_t rbytes = static_cast<size_t>(p->B * p->T * p->record_stride);
    const size_t ibytes = static_cast<size_t>(p->B * p->I * p->Sq * p->K) * (p->idx_is_i64 ? 8 : 4);
    if (overlaps(p->y, qbytes, p->q, qbytes) || overlaps(p->y, qbytes, p->k_cache, rbytes) ||
        overlaps(p->y, qbytes, p->idx, ibytes))
      return SA_ERR_OVERLAP;
    return SA_OK;
  }
  if (p->kv_dtype != p->q_dtype || dtype_bytes(p->q_dtype) == 0) return SA_ERR_DTYPE;
  if (!p->v_cache) return SA_ERR_NULL;
  if (p->Dv != p->D) return SA_ERR_UNSUPPORTED;
  if (p->B * p->Hkv * p->T >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  if (!std::isfinite(p->scale) || !std::isfinite(p->softcap) || p->softcap < 0.f)
    return SA_ERR_SHAPE;
  if (p->k_cur && (!p->v_cur || p->cur_len <= 0 || p->cur_len > p->T)) return SA_ERR_SHAPE;
  const size_t es = dtype_bytes(p->q_dtype);
  const size_t qbytes = static_cast<size_t>(p->B * p->Hq * p->Sq * p->D) * es;
  const size_t ybytes = static_cast<size_t>(p->B * p->Hq * p->Sq * p->Dv) * es;
  const size_t kvbytes = static_cast<size_t>(p->B * p->Hkv * p->T * p->D) * es;
  const size_t ibytes = static_cast<size_t>(p->B * p->I * p->Sq * p->K) * (p->idx_is_i64 ? 8 : 4);
  if (overlaps(p->y, ybytes, p->q, qbytes) || overlaps(p->y, ybytes, p->k_cache, kvbytes) ||
      overlaps(p->y, ybytes, p->v_cache, kvbytes) || overlaps(p->y, ybytes, p->idx, ibytes))
    return SA_ERR_OVERLAP;
  if ((reinterpret_cast<uintptr_t>(p->q) | reinterpret_cast<uintptr_t>(p->y)) % es) return SA_ERR_ALIGN;
  return SA_OK;
}

int sparse_plan(const sa_sparse_params* p, Plan& pl) {
  sa::GatherArgs& g = pl.g;
  memset(&g, 0, sizeof(g));
  g.q = p->q;
  g.k = p->k_cache;
  g.v = p->v_cache;
  g.y = p->y;
  g.sink = p->sink;
  g.err_word = p->err_word;
  g.source = sa::kSparse;
  if (p->bias) {
    int64_t st[4];
    bias_strides(p, st);  // checked by check_sparse
    g.bias = p->bias;
    g.bias_sb = st[0];
    g.bias_sh = st[1];
    g.bias_si = st[2];
    g.bias_sk = st[3];
  }
  g.row_copies = (p->options & SA_OPT_ROW_COPIES) ? 1 : 0;
  g.fp8_warp_mma = (p->options & SA_OPT_FP8_WARP_MMA) ? 1 : 0;
  g.B = p->B;
  g.Hq = p->Hq;
  g.Hkv = p->Hkv;
  g.Sq = p->Sq;
  g.D = p->D;
  g.Dv = p->Dv;
  g.idx = p->idx;
  g.idx_is_i64 = p->idx_is_i64;
  g.I = p->I;
  g.K = p->K;
  g.T = p->T;
  g.window = p->window;
  g.kv_len = p->kv_len;
  g.past_len = p->past_len;
  g.causal = p->causal;
  g.n_cand = p->window + p->K;
  const float scale = p->scale != 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  g.scale_log2 = scale * 1.4426950408889634f;
  g.softcap = p->softcap;
  g.inv_softcap = p->softcap != 0.f ? 1.0f / p->softcap : 0.f;
  g.k_cur = p->k_cur;
  g.v_cur = p->v_cur;
  g.write_pos = p->write_pos;
  g.C = p->k_cur ? p->cur_len : 0;
  if (p->kv_dtype == SA_FP8_E4M3_B64) {
    g.record_stride = p->record_stride;
    return plan_fp8(pl);
  }
  int rc = plan_gather(pl, p->q_dtype);
  if (rc != SA_OK) return rc;
  if (pl.stream && !(aligned16(p->k_cache) && aligned16(p->v_cache)))
    return SA_ERR_ALIGN;
  if (pl.stream && p->k_cur && !(aligned16(p->k_cur) && aligned16(p->v_cur)))
    return SA_ERR_ALIGN;
  return SA_OK;
}

}  // namespace

extern "C" {

int sa_set_kernel_events(void* before, void* after) {
  if ((before == nullptr) != (after == nullptr)) return SA_ERR_NULL;
  t_ev_before = before;
  t_ev_after = after;
  return SA_OK;
}

int sa_graph_kernel_count(void* graph) {
  if (!graph) return SA_ERR_NULL;
  cudaGraph_t g = static_cast<cudaGraph_t>(graph);
  size_t n = 0;
  if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess) return SA_ERR_LAUNCH;
  std::vector<cudaGraphNode_t> nodes(n);
  if (n > 0 && cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return SA_ERR_LAUNCH;
  int kernels = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess) return SA_ERR_LAUNCH;
    if (t == cudaGraphNodeTypeKernel) ++kernels;
  }
  return kernels;
}

int sa_check_wait_timeout(uint32_t* err_word, uint32_t* out, void* stream) {
  if (!err_word || !out) return SA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(out) % 4 || reinterpret_cast<uintptr_t>(err_word) % 4)
    return SA_ERR_ALIGN;
  return sa::launch_wait_timeout(err_word, out, static_cast<cudaStream_t>(stream)) == 0
             ? SA_OK
             : SA_ERR_LAUNCH;
}

const char* sa_status_string(int status) {
  switch (status) {
    case SA_OK: return "ok";
    case SA_ERR_NULL: return "a required pointer is NULL";
    case SA_ERR_SHAPE: return "a size is non-positive or inconsistent";
    case SA_ERR_DTYPE: return "unsupported dtype or dtype combination";
    case SA_ERR_ALIGN: return "a pointer is not suitably aligned";
    case SA_ERR_WORKSPACE: return "workspace missing or too small";
    case SA_ERR_OVERLAP: return "an output overlaps an input";
    case SA_ERR_UNSUPPORTED: return "request not served by this build";
    case SA_ERR_LAUNCH: return "CUDA launch failed";
    case SA_ERR_SCRATCH_LIMIT: return "request needs more scratch than the built-in no-allocation buffer holds";
    default: return "unknown status";
  }
}

int sa_version(void) { return 100; }

int validate_indices(const void* idx, int idx_is_i64, int64_t B, int64_t I, int64_t Sq,
                     int64_t K, const int64_t* bound_per_batch, int64_t bound,
                     uint8_t* row_status, uint32_t* err_word, void* stream) {
  if (!idx || !err_word) return SA_ERR_NULL;
  if (B <= 0 || I <= 0 || Sq <= 0 || K <= 0 || bound < 0) return SA_ERR_SHAPE;
  const size_t esz = idx_is_i64 ? 8 : 4;
  if (reinterpret_cast<uintptr_t>(idx) % esz) return SA_ERR_ALIGN;
  sa::ValidateArgs a;
  a.idx = idx;
  a.is_i64 = idx_is_i64 ? 1 : 0;
  a.vec_ok = aligned16(idx) && ((K * static_cast<int64_t>(esz)) % 16 == 0);
  a.rows = B * I * Sq;
  a.rows_per_batch = I * Sq;
  a.K = K;
  a.bound_per_batch = bound_per_batch;
  a.bound = bound;
  a.row_status = row_status;
  a.err_word = err_word;
  return sa::launch_validate(a, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

int build_present_kv(const void* past_k, const void* cur_k, void* present_k, const void* past_v,
                     const void* cur_v, void* present_v, int dtype, int64_t B, int64_t H,
                     int64_t P, int64_t C, int64_t D, int64_t present_stride,
                     const int64_t* write_pos, uint32_t* err_word, void* stream) {
  const size_t es = dtype_bytes(dtype);
  if (es == 0) return SA_ERR_DTYPE;
  if (!cur_k || !present_k) return SA_ERR_NULL;
  if (present_v && !cur_v) return SA_ERR_NULL;
  if (B <= 0 || H <= 0 || C <= 0 || D <= 0 || P < 0) return SA_ERR_SHAPE;
  sa::PresentArgs a;
  memset(&a, 0, sizeof(a));
  a.n_tensors = present_v ? 2 : 1;
  a.esz = static_cast<int>(es);
  a.B = B;
  a.H = H;
  a.P = P;
  a.C = C;
  a.D = D;
  a.stride = present_stride;
  a.write_pos = write_pos;
  a.err_word = err_word;
  const void* pasts[2] = {past_k, past_v};
  const void* curs[2] = {cur_k, cur_v};
  void* outs[2] = {present_k, present_v};
  const size_t row = static_cast<size_t>(D) * es;
  const size_t out_bytes = static_cast<size_t>(B * H * present_stride) * row;
  const size_t cur_bytes = static_cast<size_t>(B * H * C) * row;
  if (write_pos == nullptr) {
    if (present_stride < P + C) return SA_ERR_SHAPE;
    if (P > 0 && (!past_k || (present_v && !past_v))) return SA_ERR_NULL;
    const size_t past_bytes = static_cast<size_t>(B * H * P) * row;
    for (int t = 0; t < a.n_tensors; ++t) {
      for (int s = 0; s < 2; ++s) {  // against both tensors' inputs
        if (overlaps(outs[t], out_bytes, curs[s], cur_bytes) ||
            overlaps(outs[t], out_bytes, pasts[s], P > 0 ? past_bytes : 0))
          return SA_ERR_OVERLAP;
      }
    }
    if (overlaps(outs[0], out_bytes, outs[1], out_bytes)) return SA_ERR_OVERLAP;
  } else {
    if (present_stride < C) return SA_ERR_SHAPE;
    for (int t = 0; t < a.n_tensors; ++t) {
      if (pasts[t] && pasts[t] != outs[t]) {
        a.copy_past = 1;
        if (overlaps(outs[t], out_bytes, pasts[t], out_bytes)) return SA_ERR_OVERLAP;
      }
      for (int s = 0; s < a.n_tensors; ++s)
        if (overlaps(outs[t], out_bytes, curs[s], cur_bytes)) return SA_ERR_OVERLAP;
    }
    if (a.copy_past) {
      for (int t = 0; t < a.n_tensors; ++t)
        if (!pasts[t] || pasts[t] == outs[t]) return SA_ERR_UNSUPPORTED;  // mixed modes
    }
    if (overlaps(outs[0], out_bytes, outs[1], out_bytes)) return SA_ERR_OVERLAP;
  }
  for (int t = 0; t < a.n_tensors; ++t) {
    a.past[t] = pasts[t] ? pasts[t] : curs[t];
    a.cur[t] = curs[t];
    a.present[t] = outs[t];
    if (reinterpret_cast<uintptr_t>(outs[t]) % es || reinterpret_cast<uintptr_t>(curs[t]) % es)
      return SA_ERR_ALIGN;
  }
  return sa::launch_present(a, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

size_t sparse_attn_decode_workspace(const sa_sparse_params* p) {
  if (check_sparse(p, 1) != SA_OK) return 0;
  Plan pl;
  if (sparse_plan(p, pl) != SA_OK) return 0;
  return pl.bytes;
}

int sparse_attn_decode(const sa_sparse_params* p, void* stream) {
  int rc = check_sparse(p);
  if (rc != SA_OK) return rc;
  Plan pl;
  rc = sparse_plan(p, pl);
  if (rc != SA_OK) return rc;
  rc = check_workspace(pl, p->workspace, p->workspace_bytes);
  if (rc != SA_OK) return rc;
  cudaStream_t st = as_stream(stream);
  carve(pl, p->workspace);
  // Plan kernel: per index row validation + planned positions (stream path),
  // and the current-token append (either path).
  sa::PlanArgs pa;
  memset(&pa, 0, sizeof(pa));
  pa.idx = p->idx;
  pa.idx_is_i64 = p->idx_is_i64 ? 1 : 0;
  const size_t iesz = p->idx_is_i64 ? 8 : 4;
  pa.vec_ok = p->idx && aligned16(p->idx) && ((p->K * static_cast<int64_t>(iesz)) % 16 == 0);
  pa.plan_rows = (pl.stream || pl.fp8) ? 1 : 0;
  pa.write_positions = 1;
  if (pl.fp8_tc) {
    // the FP8 decode kernel plans its own positions: the plan kernel only
    // validates, beside it, when a status output is asked for
    pa.write_positions = 0;
    pa.plan_rows = (p->K > 0 && (p->err_word || p->row_status)) ? 1 : 0;
    pl.g.fp8_own_positions = 1;
    pl.g.fp8_after_plan = pa.plan_rows;
  }
  pa.validate = pa.plan_rows && p->K > 0 && (p->err_word || p->row_status);
  pa.causal = p->causal;
  pa.B = p->B;
  pa.I = p->I;
  pa.Sq = p->Sq;
  pa.K = p->K;
  pa.T = p->T;
  pa.window = p->window;
  pa.past_len = p->past_len;
  pa.n_cand_pad = pl.g.n_cand_pad;
  pa.kv_len = p->kv_len;
  pa.pos = const_cast<int32_t*>(pl.g.pos);
  pa.row_status = p->row_status;
  pa.err_word = p->err_word;
  if (p->k_cur) {
    pa.k_cur = p->k_cur;
    pa.v_cur = p->v_cur;
    pa.k_cache = const_cast<void*>(p->k_cache);
    pa.v_cache = const_cast<void*>(p->v_cache);
    pa.write_pos = p->write_pos;
    pa.Hkv = p->Hkv;
    pa.C = p->cur_len;
    pa.D = p->D;
    pa.esz = static_cast<int>(dtype_bytes(p->q_dtype));
    if ((p->D * pa.esz) % 16 || !aligned16(p->k_cur) || !aligned16(p->v_cur) ||
        !aligned16(p->k_cache) || !aligned16(p->v_cache))
      return SA_ERR_ALIGN;
    const int64_t n16 = p->B * p->Hkv * p->cur_len * (p->D * pa.esz / 16);
    int64_t blocks = (n16 + 127) / 128;
    if (blocks > 152 * 4) blocks = 152 * 4;
    pa.append_blocks = static_cast<int>(blocks);
  }
  if ((pa.plan_rows || pa.append_blocks) && sa::launch_plan(pa, st) != 0) return SA_ERR_LAUNCH;
  if (!pa.plan_rows && p->K > 0 && (p->err_word || p->row_status)) {
    sa::ValidateArgs v;
    v.idx = p->idx;
    v.is_i64 = p->idx_is_i64 ? 1 : 0;
    v.vec_ok = pa.vec_ok;
    v.rows = p->B * p->I * p->Sq;
    v.rows_per_batch = p->I * p->Sq;
    v.K = p->K;
    v.bound_per_batch = p->kv_len;
    v.bound = p->T;
    v.row_status = p->row_status;
    v.err_word = p->err_word;
    if (sa::launch_validate(v, st) != 0) return SA_ERR_LAUNCH;
  }
  return run_plan(pl, p->q_dtype, st);
}

// ---- prefill ---------------------------------------------------------------------

// [SA] mask_bias: element strides of the mask's logical axes [B, Hq, S, S]
// (0 on broadcast or missing axes) and the key-axis extent below which keys
// are kept (0: no limit).  Every axis but the last is 1 or its target.
static bool mask_layout(const sa_prefill_params* p, int64_t st[4], int64_t* key_extent) {
  const int64_t target[4] = {p->B, p->Hq, p->S, p->S};
  if (p->mask_rank < 0 || p->mask_rank > 4) return false;
  const int r = static_cast<int>(p->mask_rank);
  int64_t run = 1;
  *key_extent = 0;
  for (int ax = 3; ax >= 0; --ax) {
    const int k = ax - (4 - r);
    if (k < 0) {
      st[ax] = 0;
      continue;
    }
    const int64_t e = p->mask_dims[k];
    if (e <= 0) return false;
    if (ax < 3 && e != 1 && e != target[ax]) return false;
    if (ax == 3 && e < p->S) *key_extent = e;
    st[ax] = (e == 1) ? 0 : run;
    run *= e;
  }
  return true;
}

static int check_prefill(const sa_prefill_params* p, int query = 0) {
  if (!p || !p->q || !p->k || !p->v || (!p->y && !query)) return SA_ERR_NULL;
  if (p->reserved_ != 0) return SA_ERR_UNSUPPORTED;
  if (p->mask_kind < SA_MASK_NONE || p->mask_kind > SA_MASK_BOOL) return SA_ERR_DTYPE;
  if (p->mask_kind != SA_MASK_NONE) {
    if (!p->attn_mask) return SA_ERR_NULL;
    int64_t st[4], ke;
    if (!mask_layout(p, st, &ke)) return SA_ERR_SHAPE;
    const size_t es = p->mask_kind == SA_MASK_F32 ? 4 : p->mask_kind == SA_MASK_BOOL ? 1 : 2;
    if (reinterpret_cast<uintptr_t>(p->attn_mask) % es) return SA_ERR_ALIGN;
  }
  if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->S <= 0 || p->D <= 0) return SA_ERR_SHAPE;
  if (p->Hq % p->Hkv != 0) return SA_ERR_SHAPE;
  if (dtype_bytes(p->dtype) == 0) return SA_ERR_DTYPE;
  if (p->B * p->Hkv * p->S >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  if (!std::isfinite(p->scale) || !std::isfinite(p->softcap) || p->softcap < 0.f)
    return SA_ERR_SHAPE;
  const size_t es = dtype_bytes(p->dtype);
  const size_t qb = static_cast<size_t>(p->B * p->Hq * p->S * p->D) * es;
  const size_t kb = static_cast<size_t>(p->B * p->Hkv * p->S * p->D) * es;
  const void* ins[3] = {p->q, p->k, p->v};
  const size_t inb[3] = {qb, kb, kb};
  for (int i = 0; i < 3; ++i) {
    if (overlaps(p->y, qb, ins[i], inb[i])) return SA_ERR_OVERLAP;
    if (overlaps(p->present_k, kb, ins[i], inb[i])) return SA_ERR_OVERLAP;
    if (overlaps(p->present_v, kb, ins[i], inb[i])) return SA_ERR_OVERLAP;
  }
  if (overlaps(p->y, qb, p->present_k, kb) || overlaps(p->y, qb, p->present_v, kb) ||
      overlaps(p->present_k, kb, p->present_v, kb))
    return SA_ERR_OVERLAP;
  return SA_OK;
}

static void prefill_args(const sa_prefill_params* p, sa::GatherArgs& g) {
  memset(&g, 0, sizeof(g));
  g.q = p->q;
  g.k = p->k;
  g.v = p->v;
  g.y = p->y;
  g.source = sa::kDense;
  g.B = p->B;
  g.Hq = p->Hq;
  g.Hkv = p->Hkv;
  g.Sq = p->S;
  g.D = p->D;
  g.Dv = p->D;
  g.T = p->S;
  g.I = p->Hkv;
  g.causal = p->causal;
  g.past_len = 0;
  g.n_cand = p->S;
  const float scale = p->scale != 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  g.scale_log2 = scale * 1.4426950408889634f;
  g.softcap = p->softcap;
  g.inv_softcap = p->softcap != 0.f ? 1.0f / p->softcap : 0.f;
  g.dense_nonpad = p->nonpad_kv_seqlen;
  if (p->mask_kind != SA_MASK_NONE) {
    int64_t st[4];
    mask_layout(p, st, &g.bias_key_extent);  // checked by check_prefill
    g.bias = p->attn_mask;
    g.bias_kind = p->mask_kind == SA_MASK_F16    ? sa::kBiasF16
                  : p->mask_kind == SA_MASK_BF16 ? sa::kBiasBF16
                  : p->mask_kind == SA_MASK_BOOL ? sa::kBiasBool
                                                 : sa::kBiasF32;
    g.bias_sb = st[0];
    g.bias_sh = st[1];
    g.bias_si = st[2];
    g.bias_sk = st[3];
  }
}

static void prefill_tc_args(const sa_prefill_params* p, sa::PrefillTcArgs& a) {
  memset(&a, 0, sizeof(a));
  a.q = p->q;
  a.k = p->k;
  a.v = p->v;
  a.y = p->y;
  a.present_k = p->present_k;
  a.present_v = p->present_v;
  a.dtype = p->dtype;
  a.causal = p->causal;
  a.B = p->B;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.S = p->S;
  a.D = p->D;
  a.scale = p->scale != 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  a.softcap = p->softcap;
  a.err_word = p->err_word;
  a.nonpad = p->nonpad_kv_seqlen;
  if (a.nonpad) {  // present K/V then come from a separate copy (see attn_prefill)
    a.present_k = nullptr;
    a.present_v = nullptr;
  }
}

// Whether the tcgen05 kernel serves this call (bf16/f16, D in {64, 128},
// positive scale, 16-byte aligned q / k / v); it needs no workspace.  The
// output's alignment is not part of the choice (the workspace query has no
// output): a misaligned y on this path is SA_ERR_ALIGN.
static bool prefill_on_tc(const sa_prefill_params* p) {
  if (p->mask_kind != SA_MASK_NONE) return false;  // masks: the per-row kernels
  sa::PrefillTcArgs a;
  prefill_tc_args(p, a);
  a.y = const_cast<void*>(a.q);
  a.present_k = a.present_v = nullptr;  // checked per call, like y
  return sa::prefill_tc_supported(a);
}

size_t attn_prefill_workspace(const sa_prefill_params* p) {
  if (check_prefill(p, 1) != SA_OK) return 0;
  if (prefill_on_tc(p)) return 0;
  Plan pl;
  prefill_args(p, pl.g);
  if (plan_gather(pl, p->dtype) != SA_OK) return 0;
  return pl.bytes;
}

static int copy_present(const sa_prefill_params* p, void* stream) {
  if (!p->present_k && !p->present_v) return SA_OK;
  const void* cur_k = p->present_k ? p->k : p->v;
  void* out_k = p->present_k ? p->present_k : p->present_v;
  const void* cur_v = (p->present_k && p->present_v) ? p->v : nullptr;
  void* out_v = (p->present_k && p->present_v) ? p->present_v : nullptr;
  return build_present_kv(nullptr, cur_k, out_k, nullptr, cur_v, out_v, p->dtype, p->B, p->Hkv, 0,
                          p->S, p->D, p->S, nullptr, nullptr, stream);
}

int attn_prefill(const sa_prefill_params* p, void* stream) {
  int rc = check_prefill(p);
  if (rc != SA_OK) return rc;
  cudaStream_t st = as_stream(stream);
  if (prefill_on_tc(p)) {
    if (!aligned16(p->y) || !aligned16(p->present_k) || !aligned16(p->present_v))
      return SA_ERR_ALIGN;
    sa::PrefillTcArgs a;  // present K/V are written by the kernel itself ...
    prefill_tc_args(p, a);
    if (p->nonpad_kv_seqlen) {  // ... unless padded rows may skip their tiles
      rc = copy_present(p, stream);
      if (rc != SA_OK) return rc;
    }
    sa::mark_event(t_ev_before, st);
    const int lrc = sa::launch_prefill_tc(a, st);
    sa::mark_event(t_ev_after, st);
    return lrc == 0 ? SA_OK : SA_ERR_LAUNCH;
  }
  Plan pl;
  prefill_args(p, pl.g);
  rc = plan_gather(pl, p->dtype);
  if (rc != SA_OK) return rc;
  if (pl.stream && !(aligned16(p->k) && aligned16(p->v))) return SA_ERR_ALIGN;
  rc = check_workspace(pl, p->workspace, p->workspace_bytes);
  if (rc != SA_OK) return rc;
  rc = copy_present(p, stream);
  if (rc != SA_OK) return rc;
  carve(pl, p->workspace);
  return run_plan(pl, p->dtype, st);
}

// ---- paged decode ------------------------------------------------------------------

static int check_paged(const sa_paged_params* p, int query = 0) {
  if (!p || !p->q || !p->k_pool || !p->v_pool || !p->block_table || !p->ctx_len ||
      (!p->y && !query))
    return SA_ERR_NULL;
  if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->page_tokens <= 0 ||
      p->max_pages <= 0 || p->num_pages <= 0)
    return SA_ERR_SHAPE;
  if (p->Hq % p->Hkv != 0) return SA_ERR_SHAPE;
  if (dtype_bytes(p->dtype) == 0) return SA_ERR_DTYPE;
  if (p->options & ~SA_OPT_ROW_COPIES) return SA_ERR_UNSUPPORTED;
  if (p->num_pages * p->Hkv * p->page_tokens >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  if (!std::isfinite(p->scale)) return SA_ERR_SHAPE;
  const size_t es = dtype_bytes(p->dtype);
  const size_t yb = static_cast<size_t>(p->B * p->Hq * p->D) * es;
  const size_t pool = static_cast<size_t>(p->num_pages * p->Hkv * p->page_tokens * p->D) * es;
  if (overlaps(p->y, yb, p->q, yb) || overlaps(p->y, yb, p->k_pool, pool) ||
      overlaps(p->y, yb, p->v_pool, pool) || overlaps(p->k_pool, pool, p->v_pool, pool))
    return SA_ERR_OVERLAP;
  return SA_OK;
}

static void paged_args(const sa_paged_params* p, sa::GatherArgs& g) {
  memset(&g, 0, sizeof(g));
  g.q = p->q;
  g.k = p->k_pool;
  g.v = p->v_pool;
  g.y = p->y;
  g.err_word = p->err_word;
  g.source = sa::kPaged;
  g.B = p->B;
  g.Hq = p->Hq;
  g.Hkv = p->Hkv;
  g.Sq = 1;
  g.D = p->D;
  g.Dv = p->D;
  g.I = p->Hkv;
  g.block_table = p->block_table;
  g.ctx_len = p->ctx_len;
  g.page_tokens = p->page_tokens;
  g.max_pages = p->max_pages;
  g.num_pages = p->num_pages;
  g.n_cand = p->max_pages * p->page_tokens;
  g.row_copies = (p->options & SA_OPT_ROW_COPIES) ? 1 : 0;
  const float scale = p->scale != 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  g.scale_log2 = scale * 1.4426950408889634f;
}

size_t paged_attn_decode_workspace(const sa_paged_params* p) {
  if (check_paged(p, 1) != SA_OK) return 0;
  Plan pl;
  paged_args(p, pl.g);
  if (plan_gather(pl, p->dtype) != SA_OK) return 0;
  return pl.bytes;
}

int paged_attn_decode(const sa_paged_params* p, void* stream) {
  int rc = check_paged(p);
  if (rc != SA_OK) return rc;
  cudaStream_t st = as_stream(stream);
  Plan pl;
  paged_args(p, pl.g);
  rc = plan_gather(pl, p->dtype);
  if (rc != SA_OK) return rc;
  if (pl.stream && !(aligned16(p->k_pool) && aligned16(p->v_pool))) return SA_ERR_ALIGN;
  rc = check_workspace(pl, p->workspace, p->workspace_bytes);
  if (rc != SA_OK) return rc;
  if (p->k_new || p->v_new) {
    sa::PagedAppendArgs a;
    a.k_pool = p->k_pool;
    a.v_pool = p->v_pool;
    a.k_new = p->k_new;
    a.v_new = p->v_new;
    a.block_table = p->block_table;
    a.ctx_len = p->ctx_len;
    a.B = p->B;
    a.Hkv = p->Hkv;
    a.D = p->D;
    a.page_tokens = p->page_tokens;
    a.max_pages = p->max_pages;
    a.num_pages = p->num_pages;
    a.esz = static_cast<int>(dtype_bytes(p->dtype));
    a.err_word = p->err_word;
    if (sa::launch_paged_append(a, st) != 0) return SA_ERR_LAUNCH;
  }
  carve(pl, p->workspace);
  return run_plan(pl, p->dtype, st);
}

// ---- ratio-4 index selection -------------------------------------------------------

static int check_index(const sa_index_select_params* p, int query = 0) {
  if (!p || !p->query || !p->weight || !p->keys || (!p->selected && !query)) return SA_ERR_NULL;
  if (p->reserved_ != 0) return SA_ERR_UNSUPPORTED;
  if (p->B <= 0 || p->S <= 0 || p->IH <= 0 || p->R <= 0 || p->topk <= 0 || p->out_heads <= 0)
    return SA_ERR_SHAPE;
  if (!(p->ID == 32 || p->ID == 64 || p->ID == 128 || p->ID == 256)) return SA_ERR_UNSUPPORTED;
  if (p->IH > 256 || p->topk > 4096) return SA_ERR_UNSUPPORTED;
  if (p->key_stride < p->ID / 32 * 17 || p->key_stride % 4) return SA_ERR_SHAPE;
  if (p->key_stride * 256 > 64 * 1024) return SA_ERR_UNSUPPORTED;
  // rows up to 2^17 records (a 512K-token context at ratio 4): the
  // equal-score hash set of a row (2 R slots in 8 parts) fits in shared memory
  if (p->B * p->R >= (int64_t(1) << 31) || p->R > (int64_t(1) << 17)) return SA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(p->keys) % 4 || reinterpret_cast<uintptr_t>(p->query) % 4 ||
      reinterpret_cast<uintptr_t>(p->weight) % 4 || reinterpret_cast<uintptr_t>(p->selected) % 4)
    return SA_ERR_ALIGN;
  const size_t sbytes = static_cast<size_t>(p->B * p->out_heads * p->S * p->topk) * 4;
  const size_t qbytes = static_cast<size_t>(p->B * p->S * p->IH * p->ID) * 4;
  const size_t kbytes = static_cast<size_t>(p->B * p->R * p->key_stride);
  if (overlaps(p->selected, sbytes, p->query, qbytes) ||
      overlaps(p->selected, sbytes, p->keys, kbytes) ||
      overlaps(p->selected, sbytes, p->weight, static_cast<size_t>(p->B * p->S * p->IH) * 4))
    return SA_ERR_OVERLAP;
  return SA_OK;
}

// Workspace layout of the index selection; fills the pointers when ws != NULL.
static size_t index_plan(const sa_index_select_params* p, sa::IndexArgs& a, char* ws) {
  memset(&a, 0, sizeof(a));
  a.rows = p->B * p->S;
  a.S = p->S;
  a.IH = p->IH;
  a.ID = p->ID;
  a.R = p->R;
  a.topk = p->topk;
  a.key_stride = p->key_stride;
  a.out_heads = p->out_heads;
  int64_t slots = 2;
  while (slots < 2 * p->R) slots <<= 1;
  a.hash_slots = static_cast<int>(slots);
  int lg = 0;
  while ((int64_t(1) << lg) < slots) ++lg;
  a.hash_log2 = lg;
  int64_t sp = 1;
  while (sp < p->topk) sp <<= 1;
  a.sel_slots = static_cast<int>(sp);
  size_t off = 0;
  const size_t o_codes = off;
  off += align_up(static_cast<size_t>(a.rows * p->IH * p->ID));
  const size_t o_exp = off;
  off += align_up(static_cast<size_t>(a.rows * p->IH * (p->ID / 32)));
  const size_t o_info = off;
  off += align_up(static_cast<size_t>(a.rows * p->IH) * 16);
  const size_t o_qs = off;
  off += align_up(static_cast<size_t>(a.rows * p->IH * (p->ID / 32)) * 4);
  const size_t o_scores = off;
  off += align_up(static_cast<size_t>(a.rows * p->R) * 4);
  const size_t o_hist = off;
  off += align_up(static_cast<size_t>(a.rows) * 2048 * 4);
  const size_t o_flags = off;
  off += align_up(static_cast<size_t>(a.rows) * 4);
  const size_t o_done = off;
  off += align_up(static_cast<size_t>(a.rows) * 4);
  const size_t o_bucket = off;
  off += align_up(static_cast<size_t>(a.rows * p->R) * 8);
  if (ws) {
    a.qcodes = reinterpret_cast<int8_t*>(ws + o_codes);
    a.qexp = reinterpret_cast<int8_t*>(ws + o_exp);
    a.qinfo = reinterpret_cast<int4*>(ws + o_info);
    a.qscale = reinterpret_cast<float*>(ws + o_qs);
    a.scores = reinterpret_cast<float*>(ws + o_scores);
    a.hist = reinterpret_cast<uint32_t*>(ws + o_hist);
    a.rowflags = reinterpret_cast<uint32_t*>(ws + o_flags);
    a.done = reinterpret_cast<uint32_t*>(ws + o_done);
    a.bucket = reinterpret_cast<unsigned long long*>(ws + o_bucket);
  }
  return off;
}

size_t sparse_index_select_workspace(const sa_index_select_params* p) {
  if (check_index(p, 1) != SA_OK) return 0;
  sa::IndexArgs a;
  return index_plan(p, a, nullptr);
}

int sparse_index_select(const sa_index_select_params* p, void* stream) {
  int rc = check_index(p);
  if (rc != SA_OK) return rc;
  sa::IndexArgs a;
  const size_t need = index_plan(p, a, nullptr);
  if (!p->workspace || p->workspace_bytes < need) return SA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(p->workspace) % kAlign) return SA_ERR_ALIGN;
  index_plan(p, a, static_cast<char*>(p->workspace));
  a.query = p->query;
  a.weight = p->weight;
  a.keys = p->keys;
  a.selected = p->selected;
  a.row_status = p->row_status;
  a.err_word = p->err_word;
  a.query_start = p->query_start;
  a.query_start_b = p->query_start_b;
  a.ascending = p->ascending ? 1 : 0;
  // the pages' constants, binary32: 1/sqrt(ID), then (1/sqrt(ID))/sqrt(IH)
  const float inv_sqrt_id = 1.0f / sqrtf(static_cast<float>(p->ID));
  a.had_scale = inv_sqrt_id;
  a.weight_scale = inv_sqrt_id / sqrtf(static_cast<float>(p->IH));
  a.ev_before = t_ev_before;
  a.ev_after = t_ev_after;
  return sa::launch_index_select(a, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

// ---- compressed sparse attention, ratio 4 (the pages' own form) ------------------------

static int check_csa(const sa_csa_params* p, int query = 0) {
  if (!p || !p->query || !p->records || !p->selected || (!p->y && !query)) return SA_ERR_NULL;
  if (p->reserved_ != 0) return SA_ERR_UNSUPPORTED;
  if (p->B <= 0 || p->S <= 0 || p->H <= 0 || p->D <= 0 || p->topk <= 0 || p->R <= 0 ||
      p->L < 0 || p->total < p->S || p->n_rope < 0)
    return SA_ERR_SHAPE;
  if (p->L > 0 && !p->current_kv) return SA_ERR_NULL;
  if ((p->q_dtype != SA_F32 && p->q_dtype != SA_BF16) ||
      (p->kv_dtype != SA_F32 && p->kv_dtype != SA_BF16))
    return SA_ERR_DTYPE;
  if (!(p->D == 128 || p->D == 512) || p->H % 32 != 0) return SA_ERR_UNSUPPORTED;
  if (p->n_rope % 2 || p->n_rope >= p->D || (p->D - p->n_rope) % 64) return SA_ERR_SHAPE;
  if (p->record_stride < (p->D - p->n_rope) / 64 * 65 + 2 * p->n_rope) return SA_ERR_SHAPE;
  if (!std::isfinite(p->scale)) return SA_ERR_SHAPE;
  if (p->B * p->S * (128 + p->topk) >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  const size_t qs = p->q_dtype == SA_F32 ? 4 : 2, ks = p->kv_dtype == SA_F32 ? 4 : 2;
  if (!aligned16(p->query) || (p->current_kv && !aligned16(p->current_kv)) ||
      (p->y && !aligned16(p->y)) || reinterpret_cast<uintptr_t>(p->selected) % 4 ||
      (p->bias && reinterpret_cast<uintptr_t>(p->bias) % 4))
    return SA_ERR_ALIGN;
  if (p->bias) {
    const int64_t dense = (p->total == p->S) ? (p->L < 128 ? p->L : 128) : 128;
    const int64_t target[4] = {p->B, p->H, p->S, dense + p->topk};
    if (p->bias_rank < 0 || p->bias_rank > 4) return SA_ERR_SHAPE;
    for (int64_t r = 0; r < p->bias_rank; ++r) {
      const int64_t e = p->bias_dims[r];
      if (e != 1 && e != target[4 - p->bias_rank + r]) return SA_ERR_SHAPE;
    }
  }
  const size_t yb = static_cast<size_t>(p->B * p->S * p->H * p->D) * qs;
  if (overlaps(p->y, yb, p->query, yb) ||
      overlaps(p->y, yb, p->current_kv, static_cast<size_t>(p->B * p->L * p->D) * ks) ||
      overlaps(p->y, yb, p->records, static_cast<size_t>(p->B * p->R * p->record_stride)) ||
      overlaps(p->y, yb, p->selected, static_cast<size_t>(p->B * p->S * p->topk) * 4))
    return SA_ERR_OVERLAP;
  return SA_OK;
}

static size_t csa_plan(const sa_csa_params* p, sa::CsaArgs& a, char* ws) {
  memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.S = p->S;
  a.H = p->H;
  a.D = p->D;
  a.n_rope = p->n_rope;
  a.L = p->L;
  a.R = p->R;
  a.topk = p->topk;
  a.record_stride = p->record_stride;
  a.total = p->total;
  a.dense = (p->total == p->S) ? (p->L < 128 ? p->L : 128) : 128;
  a.valid_records = p->total / 4 < p->R ? p->total / 4 : p->R;
  const int64_t C = a.dense + p->topk;
  const int64_t sms = device_shape().sms > 0 ? device_shape().sms : 152;
  int64_t tiles, splits;
  a.tc = sa::csa_tc_supported(p->D, p->H, p->q_dtype) ? 1 : 0;
  if (a.tc) {
    // 128-slot tiles; two CTAs (halves of the output dims) per (query, 128-head
    // block, key split), one CTA per SM
    a.c_pad = (C + 127) / 128 * 128;
    tiles = a.c_pad / 128;
    const int64_t blocks = p->B * p->S * (p->H / 128) * 2;
    splits = sms / blocks;
    const int64_t min_splits = (tiles + sa::csa_tc_max_tiles() - 1) / sa::csa_tc_max_tiles();
    if (splits < min_splits) splits = min_splits;
    if (splits > 16) splits = 16 > min_splits ? 16 : min_splits;
  } else {
    a.c_pad = (C + 15) / 16 * 16;
    tiles = a.c_pad / 16;
    const int64_t blocks = p->B * p->S * (p->H / 32);
    splits = (2 * sms + blocks - 1) / blocks;  // two CTAs per SM
    if (splits > 16) splits = 16;
  }
  if (splits > tiles) splits = tiles;
  if (splits < 1) splits = 1;
  a.chunk_tiles = (tiles + splits - 1) / splits;
  a.splits = (tiles + a.chunk_tiles - 1) / a.chunk_tiles;
  const int64_t units = p->B * p->S;
  size_t off = 0;
  const size_t o_rows = off;
  off += align_up(static_cast<size_t>(units * a.c_pad * p->D) * 2);
  const size_t o_valid = off;
  off += align_up(static_cast<size_t>(units * a.c_pad));
  size_t o_po = 0, o_pml = 0;
  if (a.splits > 1) {
    o_po = off;
    off += align_up(static_cast<size_t>(units * a.splits * p->H * p->D) * 4);
    o_pml = off;
    off += align_up(static_cast<size_t>(units * a.splits * p->H) * 8);
  }
  if (ws) {
    a.rows = reinterpret_cast<__nv_bfloat16*>(ws + o_rows);
    a.valid = reinterpret_cast<uint8_t*>(ws + o_valid);
    if (a.splits > 1) {
      a.part_o = reinterpret_cast<float*>(ws + o_po);
      a.part_ml = reinterpret_cast<float*>(ws + o_pml);
    }
  }
  return off;
}

size_t csa_ratio4_attention_workspace(const sa_csa_params* p) {
  if (check_csa(p, 1) != SA_OK) return 0;
  sa::CsaArgs a;
  return csa_plan(p, a, nullptr);
}

int csa_ratio4_attention(const sa_csa_params* p, void* stream) {
  int rc = check_csa(p);
  if (rc != SA_OK) return rc;
  sa::CsaArgs a;
  const size_t need = csa_plan(p, a, nullptr);
  if (!p->workspace || p->workspace_bytes < need) return SA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(p->workspace) % kAlign) return SA_ERR_ALIGN;
  csa_plan(p, a, static_cast<char*>(p->workspace));
  a.query = p->query;
  a.window = p->current_kv;
  a.records = p->records;
  a.selected = p->selected;
  a.sink = p->sink;
  a.y = p->y;
  a.q_dtype = p->q_dtype;
  a.kv_dtype = p->kv_dtype;
  a.err_word = p->err_word;
  const float scale = p->scale != 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  a.scale_log2 = scale * 1.4426950408889634f;
  if (p->bias) {
    // right-aligned strides against [B, H, S, C] (0 on broadcast or missing axes)
    int64_t st[4] = {0, 0, 0, 0};
    int64_t run = 1;
    for (int ax = 3; ax >= 0; --ax) {
      const int k = ax - (4 - static_cast<int>(p->bias_rank));
      if (k < 0) continue;
      const int64_t e = p->bias_dims[k];
      st[ax] = (e == 1) ? 0 : run;
      run *= e;
    }
    a.bias = p->bias;
    a.bias_sb = st[0];
    a.bias_sh = st[1];
    a.bias_si = st[2];
    a.bias_sk = st[3];
  }
  a.ev_before = t_ev_before;
  a.ev_after = t_ev_after;
  return sa::launch_csa(a, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

// ---- CSA compression stages ------------------------------------------------------------

static int check_compress(const sa_compress_params* p, int ratio, int kind) {
  if (!p || !p->ape || !p->norm || !p->carry) return SA_ERR_NULL;
  if (!p->records && !p->logical) return SA_ERR_NULL;
  if (p->reserved_ != 0) return SA_ERR_UNSUPPORTED;
  if (p->B <= 0 || p->S < 0 || p->D <= 0 || p->total < p->S || p->n_rope < 0 || p->rows < 0)
    return SA_ERR_SHAPE;
  if (p->S > 0 && (!p->kv || !p->gate)) return SA_ERR_NULL;
  if (p->n_rope % 2 || p->n_rope > p->D || p->n_rope > 128) return SA_ERR_SHAPE;
  if (kind == sa::kCompressAttn) {
    if (p->D % 4 || p->D > 1024 || (p->D - p->n_rope) % 64) return SA_ERR_SHAPE;
  } else if (!(p->D == 32 || p->D == 64 || p->D == 128 || p->D == 256)) {
    return SA_ERR_SHAPE;
  }
  if (p->rows < p->total / ratio) return SA_ERR_SHAPE;
  const int64_t width = kind == sa::kCompressAttn
                            ? (p->D - p->n_rope) / 64 * 65 + 2 * p->n_rope
                            : p->D / 32 * 17;
  if (p->records && p->record_stride < width) return SA_ERR_SHAPE;
  const int64_t W = ratio == 4 ? 2 * p->D : p->D;
  const int64_t slots = ratio == 4 ? 8 : 128;
  // index arithmetic stays in 64 bits; grids need the counts below 2^31
  if (p->total / ratio - (p->total - p->S) / ratio >= (int64_t(1) << 31) ||
      p->B >= (int64_t(1) << 31) || p->total >= (int64_t(1) << 53))
    return SA_ERR_UNSUPPORTED;
  if (!aligned16(p->kv) || !aligned16(p->gate) || !aligned16(p->ape) || !aligned16(p->carry) ||
      reinterpret_cast<uintptr_t>(p->norm) % 4 || reinterpret_cast<uintptr_t>(p->logical) % 4 ||
      reinterpret_cast<uintptr_t>(p->err_word) % 4)
    return SA_ERR_ALIGN;
  const size_t carry_b = static_cast<size_t>(p->B * slots * 2 * W) * 4;
  const size_t src_b = static_cast<size_t>(p->B * p->S * W) * 4;
  const size_t rec_b = p->records ? static_cast<size_t>(p->B * p->rows * p->record_stride) : 0;
  const size_t log_b = p->logical ? static_cast<size_t>(p->B * p->rows * p->D) * 4 : 0;
  if (overlaps(p->carry, carry_b, p->kv, src_b) || overlaps(p->carry, carry_b, p->gate, src_b) ||
      overlaps(p->records, rec_b, p->carry, carry_b) ||
      overlaps(p->logical, log_b, p->carry, carry_b) ||
      overlaps(p->records, rec_b, p->logical, log_b) ||
      overlaps(p->records, rec_b, p->kv, src_b) || overlaps(p->logical, log_b, p->kv, src_b) ||
      overlaps(p->records, rec_b, p->gate, src_b) || overlaps(p->logical, log_b, p->gate, src_b))
    return SA_ERR_OVERLAP;
  return SA_OK;
}

static int compress_entry(const sa_compress_params* p, void* stream, int ratio, int kind) {
  const int rc = check_compress(p, ratio, kind);
  if (rc != SA_OK) return rc;
  sa::CompressArgs a;
  memset(&a, 0, sizeof(a));
  a.kv = p->kv;
  a.gate = p->gate;
  a.ape = p->ape;
  a.norm = p->norm;
  a.carry = p->carry;
  a.records = p->records;
  a.logical = p->logical;
  a.err_word = p->err_word;
  a.B = p->B;
  a.S = p->S;
  a.D = static_cast<int>(p->D);
  a.W = ratio == 4 ? 2 * p->D : p->D;
  a.rows = p->rows;
  a.record_stride = p->record_stride;
  a.total = p->total;
  a.start = p->total - p->S;
  a.ratio = ratio;
  a.kind = kind;
  a.n_rope = static_cast<int>(p->n_rope);
  a.width = static_cast<int>(kind == sa::kCompressAttn
                                 ? (p->D - p->n_rope) / 64 * 65 + 2 * p->n_rope
                                 : p->D / 32 * 17);
  a.k0 = a.start / ratio;
  a.nk = p->total / ratio - a.k0;
  for (int64_t i = 0; i < p->n_rope / 2; ++i) {
    // the base frequency of pair i: a binary32 exponent, the power rounded once
    const float ex = -static_cast<float>(2 * i) / static_cast<float>(p->n_rope);
    a.rope_base[i] = static_cast<float>(std::pow(160000.0, static_cast<double>(ex)));
  }
  a.ev_before = t_ev_before;
  a.ev_after = t_ev_after;
  return sa::launch_compress(a, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

int csa_ratio128_compress(const sa_compress_params* p, void* stream) {
  return compress_entry(p, stream, 128, sa::kCompressAttn);
}

int csa_ratio4_main_compress(const sa_compress_params* p, void* stream) {
  return compress_entry(p, stream, 4, sa::kCompressAttn);
}

int csa_ratio4_index_compress(const sa_compress_params* p, void* stream) {
  return compress_entry(p, stream, 4, sa::kCompressIndex);
}

int csa_pool_weight(const float* t, float* w, int64_t n, void* stream) {
  if (n < 0) return SA_ERR_SHAPE;
  if (n > 0 && (!t || !w)) return SA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(t) % 4 || reinterpret_cast<uintptr_t>(w) % 4)
    return SA_ERR_ALIGN;
  return sa::launch_pool_weight(t, w, n, as_stream(stream)) == 0 ? SA_OK : SA_ERR_LAUNCH;
}

}  // extern "C"

// ---- sparse decode without caller-provided scratch ------------------------------------
//
// For callers that may not allocate device memory: a runtime that owns a fixed
// device-memory budget and accounts for every byte, a plugin whose host
// framework hands it inputs and outputs but no scratch, or code that must not
// trigger cudaMalloc's implicit device synchronisation (or its refusal during
// a global-mode stream capture).  The scratch lives in one file-scope device
// array that every GPU loading this library holds until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // SA_NOALLOC_SCRATCH_BYTES
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked up
// once per device (with that device current) and cached.
void* noalloc_scratch(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = SA_ERR_LAUNCH;
    return nullptr;
  }
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      *status = SA_ERR_LAUNCH;
      return nullptr;
    }
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" int sparse_attn_decode_noalloc(const sa_sparse_params* p, void* stream) {
  int rc = check_sparse(p);
  if (rc != SA_OK) return rc;
  Plan pl;
  rc = sparse_plan(p, pl);
  if (rc != SA_OK) return rc;
  if (pl.bytes > kNoAllocScratchBytes) return SA_ERR_SCRATCH_LIMIT;
  void* scratch = noalloc_scratch(&rc);
  if (!scratch) return rc;
  sa_sparse_params q = *p;
  q.workspace = scratch;
  q.workspace_bytes = kNoAllocScratchBytes;
  return sparse_attn_decode(&q, stream);
}
