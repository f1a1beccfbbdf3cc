/*
 * sa_oracle.c -- plain, slow, fp64 CPU oracle for KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library: storage decoding, FP8 decoding, index validation, present-KV
 * construction and attention are all written out again here, directly from
 * the definitions, with no blocking, fusion or reordering.
 *
 * Sources (the pages' titles and sections):
 *   [IS]  onnx-runtime-ep-cuda, src/kernels/index_share.rs -- IndexShare:
 *         module docs (selected-token attention), `validate_indices`,
 *         `build_present`, `index_share_row`.
 *   [SA]  onnx-runtime-ep-cuda, src/kernels/standard_attention.rs -- ONNX
 *         Attention: module docs "Semantics", `attention_row`,
 *         `attention_combine` (fully-masked row gives 0).
 *   [CSA] onnx-runtime-ep-cpu, src/kernels/compressed_sparse_attention.rs --
 *         `CacheFormat` (hybrid FP8 record), `dequantize_cache`; and
 *         onnx-runtime-ep-cuda compressed_sparse_attention.rs,
 *         `csa_ratio128_sink_attention` (dense window + records, sink).
 *   [PG]  ferrum-kernels, vnext_ops/transformer/causal_attention.rs --
 *         16-token KV blocks addressed through a table.
 *   [IS] `bias_at` and `validate_bias_shape`: the optional additive bias of a
 *         selected-token score, a tensor of rank <= 4 broadcast right-aligned
 *         against [batch, q_head, query, cache position].
 *   [SA] `mask_bias` and the padding frontier (`nonpad_kv_seqlen`) of
 *         `attention_row`: the attention mask and the causal offset.
 *   [CSA-CPU] compress_ratio4_stream, pool_ratio4_record,
 *         pool_ratio128_record, finalize_attention_record,
 *         finalize_index_record, apply_compressed_rope: the compression
 *         stages that produce the records.
 *   OCP 8-bit floating point specification (E4M3FN) and the OCP MX
 *   specification (E8M0 scale) for the FP8 record decode.
 *
 * Every floating-point step of the attention runs in double.  Inputs are
 * widened exactly from their storage type (f32, f16, bf16, FP8 record).  The
 * index selection and the compression stages produce bytes that the pages
 * fix in binary32, so those sections follow the pages' binary32 steps.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2
#define ORC_FP8REC 3

/* ------------------------------------------------------------------------ */
/* Exact widening of storage types.                                          */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1f;
  int fr = h & 0x3ff;
  double v;
  if (ex == 0) {
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^-14 * 2^-10 */
  } else if (ex == 31) {
    v = fr ? NAN : INFINITY;
  } else {
    v = ldexp((double)(fr | 0x400), ex - 25); /* 1.fr * 2^(ex-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double load_elem(const void* base, int64_t i, int dtype) {
  if (dtype == ORC_F32) {
    return (double)((const float*)base)[i];
  }
  if (dtype == ORC_F16) {
    return orc_f16_to_double(((const uint16_t*)base)[i]);
  }
  return orc_bf16_to_double(((const uint16_t*)base)[i]);
}

/* OCP E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinity;
 * S.1111.111 is NaN; exponent field 0 is subnormal m * 2^-9. */
double orc_e4m3fn_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int ex = (c >> 3) & 0xf;
  int m = c & 0x7;
  double v;
  if (ex == 0xf && m == 0x7) {
    return NAN;
  }
  if (ex == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp((double)(8 + m), ex - 10); /* (1 + m/8) * 2^(ex-7) */
  }
  return sign ? -v : v;
}

/* OCP MX E8M0 scale: 2^(b - 127); 0xFF is NaN. */
double orc_e8m0_to_double(uint8_t b) {
  if (b == 0xff) {
    return NAN;
  }
  return ldexp(1.0, (int)b - 127);
}

/* Decode one hybrid FP8 record into `out[n_nope + n_rope]`:
 * n_nope/64 blocks of [E8M0 scale byte, 64 E4M3FN codes], then n_rope
 * little-endian bf16 values ([CSA] CacheFormat::Fp8E4m3Block64 and
 * dequantize_cache). */
void orc_decode_fp8_record(const uint8_t* rec, int64_t n_nope, int64_t n_rope, double* out) {
  int64_t nb = n_nope / 64;
  for (int64_t blk = 0; blk < nb; ++blk) {
    const uint8_t* p = rec + blk * 65;
    double s = orc_e8m0_to_double(p[0]);
    for (int64_t d = 0; d < 64; ++d) {
      out[blk * 64 + d] = orc_e4m3fn_to_double(p[1 + d]) * s;
    }
  }
  const uint8_t* tail = rec + nb * 65;
  for (int64_t r = 0; r < n_rope; ++r) {
    uint16_t bits = (uint16_t)(tail[2 * r] | ((uint16_t)tail[2 * r + 1] << 8));
    out[n_nope + r] = orc_bf16_to_double(bits);
  }
}

/* ------------------------------------------------------------------------ */
/* Index validation ([IS] validate_indices).                                 */
/* ------------------------------------------------------------------------ */

#define ORC_IDX_OK 0
#define ORC_IDX_BELOW_SENTINEL 1
#define ORC_IDX_AFTER_PADDING 2
#define ORC_IDX_OUT_OF_RANGE 4
#define ORC_IDX_NOT_INCREASING 8
#define ORC_IDX_DUPLICATE 16
#define ORC_IDX_ALL_PADDING 32

static int64_t load_index(const void* idx, int64_t i, int is_i64) {
  return is_i64 ? ((const int64_t*)idx)[i] : (int64_t)((const int32_t*)idx)[i];
}

/* Scan one row left to right.  A -1 marks padding and is skipped; any other
 * value is checked in this order: below the -1 sentinel, after padding, out
 * of [0, bound), equal to the previous kept index, smaller than it.  The first
 * failing column decides the status.  A row with no kept index is all
 * padding. */
int orc_validate_row(const void* row, int is_i64, int64_t K, int64_t bound,
                     int64_t* bad_col) {
  int padding = 0;
  int have_prev = 0;
  int64_t prev = 0;
  int64_t count = 0;
  for (int64_t col = 0; col < K; ++col) {
    int64_t v = load_index(row, col, is_i64);
    int code = ORC_IDX_OK;
    if (v == -1) {
      padding = 1;
      continue;
    }
    if (v < -1) {
      code = ORC_IDX_BELOW_SENTINEL;
    } else if (padding) {
      code = ORC_IDX_AFTER_PADDING;
    } else if (v >= bound) {
      code = ORC_IDX_OUT_OF_RANGE;
    } else if (have_prev && v == prev) {
      code = ORC_IDX_DUPLICATE;
    } else if (have_prev && v < prev) {
      code = ORC_IDX_NOT_INCREASING;
    }
    if (code != ORC_IDX_OK) {
      if (bad_col) {
        *bad_col = col;
      }
      return code;
    }
    prev = v;
    have_prev = 1;
    count += 1;
  }
  if (count == 0) {
    if (bad_col) {
      *bad_col = -1;
    }
    return ORC_IDX_ALL_PADDING;
  }
  if (bad_col) {
    *bad_col = -1;
  }
  return ORC_IDX_OK;
}

/* Rows are [B, I, Sq] of K columns; batch b is bounded by bound_b[b] when
 * given, else by `bound`.  Fills status[row] and ORs every status into *err. */
void orc_validate_indices(const void* idx, int is_i64, int64_t B, int64_t I, int64_t Sq,
                          int64_t K, const int64_t* bound_b, int64_t bound,
                          uint8_t* status, uint32_t* err) {
  uint32_t acc = 0;
  for (int64_t b = 0; b < B; ++b) {
    int64_t bnd = bound_b ? bound_b[b] : bound;
    for (int64_t h = 0; h < I; ++h) {
      for (int64_t q = 0; q < Sq; ++q) {
        int64_t row = (b * I + h) * Sq + q;
        const char* base = (const char*)idx + row * K * (is_i64 ? 8 : 4);
        int s = orc_validate_row(base, is_i64, K, bnd, NULL);
        if (status) {
          status[row] = (uint8_t)s;
        }
        acc |= (uint32_t)s;
      }
    }
  }
  if (err) {
    *err = acc;
  }
}

/* ------------------------------------------------------------------------ */
/* Present KV ([IS] build_present; [SA] build_kv capacity append).           */
/* ------------------------------------------------------------------------ */

/* present[b,h,t,:] = past[b,h,t,:] for t < P, cur[b,h,t-P,:] for P <= t < P+C;
 * present rows have stride `out_stride` positions (>= P+C).  Byte copy of
 * `esz`-byte elements. */
void orc_present_concat(const void* past, const void* cur, void* out, int64_t esz,
                        int64_t B, int64_t H, int64_t P, int64_t C, int64_t D,
                        int64_t out_stride) {
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      for (int64_t t = 0; t < P + C; ++t) {
        const char* src;
        if (t < P) {
          src = (const char*)past + (((b * H + h) * P + t) * D) * esz;
        } else {
          src = (const char*)cur + (((b * H + h) * C + (t - P)) * D) * esz;
        }
        char* dst = (char*)out + (((b * H + h) * out_stride + t) * D) * esz;
        memcpy(dst, src, (size_t)(D * esz));
      }
    }
  }
}

/* Append: cache[b,h,write_pos[b]+c,:] = cur[b,h,c,:]; all other positions of
 * the capacity-`cap` cache are left as they are. */
void orc_present_append(const void* cur, void* cache, int64_t esz, int64_t B, int64_t H,
                        int64_t C, int64_t D, int64_t cap, const int64_t* write_pos) {
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      for (int64_t c = 0; c < C; ++c) {
        int64_t t = write_pos[b] + c;
        const char* src = (const char*)cur + (((b * H + h) * C + c) * D) * esz;
        char* dst = (char*)cache + (((b * H + h) * cap + t) * D) * esz;
        memcpy(dst, src, (size_t)(D * esz));
      }
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Attention over an explicit candidate key set.                             */
/* ------------------------------------------------------------------------ */

/* KV storage accessor: either a dense [B, Hkv, stride, D] tensor of f32/f16/
 * bf16, or hybrid FP8 records [B, Hkv, stride, record_bytes] where K and V are
 * the same decoded record (V optionally its first Dv dims). */
typedef struct {
  const void* k;
  const void* v;
  int dtype;
  int64_t Hkv;
  int64_t stride;       /* positions between consecutive (b, kvh) slabs */
  int64_t D;
  int64_t Dv;
  int64_t record_bytes; /* FP8 only */
  int64_t n_rope;       /* FP8 only */
} orc_kv;

static void get_k(const orc_kv* kv, int64_t b, int64_t h, int64_t t, double* out) {
  if (kv->dtype == ORC_FP8REC) {
    const uint8_t* rec = (const uint8_t*)kv->k +
                         ((b * kv->Hkv + h) * kv->stride + t) * kv->record_bytes;
    orc_decode_fp8_record(rec, kv->D - kv->n_rope, kv->n_rope, out);
    return;
  }
  int64_t base = ((b * kv->Hkv + h) * kv->stride + t) * kv->D;
  for (int64_t d = 0; d < kv->D; ++d) {
    out[d] = load_elem(kv->k, base + d, kv->dtype);
  }
}

static void get_v(const orc_kv* kv, int64_t b, int64_t h, int64_t t, double* out,
                  double* tmp) {
  if (kv->dtype == ORC_FP8REC) {
    const uint8_t* rec = (const uint8_t*)kv->v +
                         ((b * kv->Hkv + h) * kv->stride + t) * kv->record_bytes;
    orc_decode_fp8_record(rec, kv->D - kv->n_rope, kv->n_rope, tmp);
    for (int64_t d = 0; d < kv->Dv; ++d) {
      out[d] = tmp[d];
    }
    return;
  }
  int64_t base = ((b * kv->Hkv + h) * kv->stride + t) * kv->Dv;
  for (int64_t d = 0; d < kv->Dv; ++d) {
    out[d] = load_elem(kv->v, base + d, kv->dtype);
  }
}

/* One output row ([SA] Semantics; [IS] index_share_row):
 *   s_j = scale * sum_d q_d k_{j,d}
 *   s_j = softcap * tanh(s_j / softcap)            if softcap != 0
 *   s_j = s_j + bias[j]                              if a bias is given
 *   s_j = -inf  if masked[j]                         (causal / pad / not a key)
 *   M = max_j s_j;  M == -inf  =>  y = 0
 *   L = sum_j exp(s_j - M)  (+ exp(sink - M) if a sink logit is given)
 *   y = sum_j exp(s_j - M) / L * v_j
 * `keys` lists n candidate positions, `masked` flags the ones that take -inf.
 */
static void attend_row(const orc_kv* kv, int64_t b, int64_t kvh, const double* q,
                       const int64_t* keys, const int* masked, int64_t n, double scale,
                       double softcap, const double* bias, const double* sink, double* y) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* krow = (double*)malloc(sizeof(double) * (size_t)kv->D);
  double* vrow = (double*)malloc(sizeof(double) * (size_t)kv->D);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)kv->D);
  double M = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    if (masked[j]) {
      s[j] = -INFINITY;
      continue;
    }
    get_k(kv, b, kvh, keys[j], krow);
    double dot = 0.0;
    for (int64_t d = 0; d < kv->D; ++d) {
      dot += q[d] * krow[d];
    }
    double sj = scale * dot;
    if (softcap != 0.0) {
      sj = softcap * tanh(sj / softcap);
    }
    if (bias) {
      sj += bias[j];
    }
    s[j] = sj;
    if (sj > M) {
      M = sj;
    }
  }
  for (int64_t d = 0; d < kv->Dv; ++d) {
    y[d] = 0.0;
  }
  if (M == -INFINITY) {
    free(s);
    free(krow);
    free(vrow);
    free(tmp);
    return;
  }
  double L = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    if (s[j] != -INFINITY) {
      L += exp(s[j] - M);
    }
  }
  if (sink) {
    L += exp(*sink - M);
  }
  for (int64_t j = 0; j < n; ++j) {
    if (s[j] == -INFINITY) {
      continue;
    }
    double p = exp(s[j] - M) / L;
    get_v(kv, b, kvh, keys[j], vrow, tmp);
    for (int64_t d = 0; d < kv->Dv; ++d) {
      y[d] += p * vrow[d];
    }
  }
  free(s);
  free(krow);
  free(vrow);
  free(tmp);
}

/* ------------------------------------------------------------------------ */
/* Sparse selected-token decode ([IS] index_share_row; [CSA] window).        */
/* ------------------------------------------------------------------------ */

typedef struct {
  const void* q;        /* [B, Hq, Sq, D] in q_dtype */
  int q_dtype;          /* f32 / f16 / bf16 */
  const void* k;        /* dense: [B, Hkv, T, D]; FP8: records [B, Hkv, T, rb] */
  const void* v;        /* dense: [B, Hkv, T, Dv]; FP8: same records as k */
  int kv_dtype;         /* f32 / f16 / bf16 / FP8 record */
  const void* idx;      /* [B, I, Sq, K] */
  int idx_is_i64;
  int64_t B, Hq, Hkv, Sq, D, Dv, T, I, K;
  const int64_t* kv_len; /* nullable: per-batch valid length (pad frontier) */
  int64_t past_len;     /* causal frontier offset: query i sees j <= past_len + i */
  int causal;
  double scale;
  double softcap;
  int64_t window;       /* 0, or W: the W positions before the valid length */
  const double* sink;   /* nullable: per-query-head logit added to the denominator */
  int64_t record_bytes; /* FP8 only */
  int64_t n_rope;       /* FP8 only */
  const float* bias;    /* nullable: additive bias of rank bias_rank (<= 4) */
  int64_t bias_rank;
  int64_t bias_dims[4]; /* its shape, the first bias_rank entries */
} orc_sparse_args;

/* [IS] bias_at: the bias entry of logical element (b, h, i, j).  The bias
 * shape lines up with [B, Hq, Sq, T] from the right; an axis of extent 1 is
 * broadcast (index 0), any other axis is indexed by the logical coordinate;
 * the offset is row-major over the bias's own shape. */
static double orc_bias_at(const float* bias, int64_t rank, const int64_t* dims, int64_t b,
                          int64_t h, int64_t i, int64_t j) {
  int64_t logical[4] = {b, h, i, j};
  int64_t off = 0;
  for (int64_t r = 0; r < rank; ++r) {
    int64_t axis = 4 - rank + r;
    int64_t extent = dims[r];
    int64_t index = (extent == 1) ? 0 : logical[axis];
    off = off * extent + index;
  }
  return (double)bias[off];
}

/* [IS] validate_bias_shape: rank <= 4 and every axis 1 or equal to the
 * matching axis of [B, Hq, Sq, T] counted from the right. */
static int orc_bias_shape_ok(const orc_sparse_args* a) {
  int64_t target[4] = {a->B, a->Hq, a->Sq, a->T};
  if (a->bias_rank < 0 || a->bias_rank > 4) {
    return 0;
  }
  for (int64_t r = 0; r < a->bias_rank; ++r) {
    int64_t want = target[4 - a->bias_rank + r];
    if (a->bias_dims[r] != 1 && a->bias_dims[r] != want) {
      return 0;
    }
  }
  return 1;
}

/* Candidate set of one row:
 *   the valid prefix of idx[b, ih, i, :] (take while != -1), and with a
 *   window W additionally every t in [len_b - W, len_b), the selected entries
 *   then being kept only below len_b - W so that each key counts once.
 * A kept key is masked when causal and j > past_len + i, or when j >= len_b.
 * With a bias, the score of key j gains bias(b, h, i, j) after the softcap
 * ([IS] index_share_row adds it to the scaled score; the key is the cache
 * position); a -inf entry masks the key.
 * Rows are flattened (b, h, i); `rows` selects which to compute (NULL: all),
 * y gets one Dv-vector per computed row.  Returns 0, or -1 on a bad shape. */
int orc_sparse_attention(const orc_sparse_args* a, const int64_t* rows, int64_t nrows,
                         double* y) {
  if (a->Hkv <= 0 || a->Hq % a->Hkv != 0) {
    return -1;
  }
  if (!(a->I == 1 || a->I == a->Hkv || a->I == a->Hq)) {
    return -1;
  }
  if (a->bias && !orc_bias_shape_ok(a)) {
    return -1;
  }
  int64_t g = a->Hq / a->Hkv;
  int64_t total = a->B * a->Hq * a->Sq;
  int64_t count = rows ? nrows : total;
  orc_kv kv = {a->k, a->v, a->kv_dtype, a->Hkv, a->T, a->D, a->Dv, a->record_bytes,
               a->n_rope};
  int64_t cap = a->K + a->window;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
  int* masked = (int*)malloc(sizeof(int) * (size_t)(cap > 0 ? cap : 1));
  double* brow = (double*)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
  double* q = (double*)malloc(sizeof(double) * (size_t)a->D);
  for (int64_t r = 0; r < count; ++r) {
    int64_t row = rows ? rows[r] : r;
    int64_t i = row % a->Sq;
    int64_t h = (row / a->Sq) % a->Hq;
    int64_t b = row / (a->Sq * a->Hq);
    int64_t kvh = h / g;
    int64_t ih = (a->I == 1) ? 0 : (a->I == a->Hkv ? kvh : h);
    int64_t len = a->kv_len ? a->kv_len[b] : a->T;
    for (int64_t d = 0; d < a->D; ++d) {
      q[d] = load_elem(a->q, ((b * a->Hq + h) * a->Sq + i) * a->D + d, a->q_dtype);
    }
    int64_t n = 0;
    int64_t wstart = len - a->window;
    if (a->window > 0) {
      for (int64_t t = (wstart > 0 ? wstart : 0); t < len; ++t) {
        keys[n++] = t;
      }
    }
    const char* irow = (const char*)a->idx +
                       (((b * a->I + ih) * a->Sq + i) * a->K) * (a->idx_is_i64 ? 8 : 4);
    for (int64_t c = 0; c < a->K; ++c) {
      int64_t j = load_index(irow, c, a->idx_is_i64);
      if (j == -1) {
        break;
      }
      if (a->window > 0 && j >= wstart) {
        continue;
      }
      keys[n++] = j;
    }
    for (int64_t j = 0; j < n; ++j) {
      int m = 0;
      if (a->causal && keys[j] > a->past_len + i) {
        m = 1;
      }
      if (keys[j] >= len || keys[j] < 0) {
        m = 1;
      }
      masked[j] = m;
      brow[j] = 0.0;
      if (a->bias && !m) {
        brow[j] = orc_bias_at(a->bias, a->bias_rank, a->bias_dims, b, h, i, keys[j]);
      }
    }
    attend_row(&kv, b, kvh, q, keys, masked, n, a->scale, a->softcap, a->bias ? brow : NULL,
               a->sink ? &a->sink[h] : NULL, y + r * a->Dv);
  }
  free(keys);
  free(masked);
  free(brow);
  free(q);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Dense prefill ([SA] Semantics, attention_row), no past.                   */
/* ------------------------------------------------------------------------ */

/* [SA] mask_bias: the attention-mask term of logical element (b, h, i, j).
 * The mask's shape lines up with [B, Hq, S, S] from the right (an axis of 1
 * broadcasts).  The last axis is the key axis: a key j at or past its extent
 * takes -inf (so a last axis shorter than S, 1 included, pads with -inf); a bool mask keeps a key where it is nonzero (term 0) and masks it
 * where it is zero (-inf); f32 / f16 / bf16 masks add their value. */
#define ORC_MASK_NONE 0
#define ORC_MASK_F32 1
#define ORC_MASK_F16 2
#define ORC_MASK_BF16 3
#define ORC_MASK_BOOL 4
static double orc_mask_at(const void* mask, int kind, int64_t rank, const int64_t* dims,
                          int64_t b, int64_t h, int64_t i, int64_t j) {
  int64_t logical[4] = {b, h, i, j};
  int64_t off = 0;
  if (rank > 0 && j >= dims[rank - 1]) { /* (an extent of 1 included) */
    return -INFINITY;
  }
  for (int64_t r = 0; r < rank; ++r) {
    int64_t axis = 4 - rank + r;
    int64_t extent = dims[r];
    int64_t index = (extent == 1) ? 0 : logical[axis];
    off = off * extent + index;
  }
  switch (kind) {
    case ORC_MASK_F32:
      return (double)((const float*)mask)[off];
    case ORC_MASK_F16:
      return orc_f16_to_double(((const uint16_t*)mask)[off]);
    case ORC_MASK_BF16:
      return orc_bf16_to_double(((const uint16_t*)mask)[off]);
    case ORC_MASK_BOOL:
      return ((const uint8_t*)mask)[off] != 0 ? 0.0 : -INFINITY;
    default:
      return 0.0;
  }
}

typedef struct {
  const void* mask;          /* nullable */
  int kind;                  /* ORC_MASK_* */
  int64_t rank;
  int64_t dims[4];
  const int64_t* nonpad;     /* nullable: per-batch valid key count */
} orc_prefill_mask;

/* Q [B, Hq, S, D], K/V [B, Hkv, S, D] ([SA] Semantics, attention_row, no
 * past).  Keys j >= nonpad[b] are masked (the padding frontier) when nonpad
 * is given; when causal, query i sees keys j <= i + offset with offset =
 * nonpad[b] - S (0 without nonpad), so a row with i + offset < 0 is fully
 * masked; the mask term is added after the softcap.  Rows flattened
 * (b, h, i). */
int orc_prefill_masked(const void* q, const void* k, const void* v, int dtype, int64_t B,
                       int64_t Hq, int64_t Hkv, int64_t S, int64_t D, int causal, double scale,
                       double softcap, const orc_prefill_mask* mk, const int64_t* rows,
                       int64_t nrows, double* y) {
  if (Hkv <= 0 || Hq % Hkv != 0) {
    return -1;
  }
  int64_t g = Hq / Hkv;
  int64_t total = B * Hq * S;
  int64_t count = rows ? nrows : total;
  orc_kv kv = {k, v, dtype, Hkv, S, D, D, 0, 0};
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)S);
  int* masked = (int*)malloc(sizeof(int) * (size_t)S);
  double* brow = (double*)malloc(sizeof(double) * (size_t)S);
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  int with_mask = mk && mk->mask && mk->kind != ORC_MASK_NONE;
  for (int64_t r = 0; r < count; ++r) {
    int64_t row = rows ? rows[r] : r;
    int64_t i = row % S;
    int64_t h = (row / S) % Hq;
    int64_t b = row / (S * Hq);
    int64_t pad = (mk && mk->nonpad) ? mk->nonpad[b] : -1;
    int64_t offset = (mk && mk->nonpad) ? mk->nonpad[b] - S : 0;
    for (int64_t d = 0; d < D; ++d) {
      qr[d] = load_elem(q, ((b * Hq + h) * S + i) * D + d, dtype);
    }
    for (int64_t j = 0; j < S; ++j) {
      keys[j] = j;
      int m = 0;
      if (pad >= 0 && j >= pad) {
        m = 1;
      }
      if (causal && j > i + offset) {
        m = 1;
      }
      masked[j] = m;
      brow[j] = (with_mask && !m) ? orc_mask_at(mk->mask, mk->kind, mk->rank, mk->dims, b, h, i, j)
                                  : 0.0;
    }
    attend_row(&kv, b, h / g, qr, keys, masked, S, scale, softcap, with_mask ? brow : NULL, NULL,
               y + r * D);
  }
  free(keys);
  free(masked);
  free(brow);
  free(qr);
  return 0;
}

/* Q [B, Hq, S, D], K/V [B, Hkv, S, D]; query i sees keys 0..i when causal,
 * all S keys otherwise.  Rows flattened (b, h, i). */
int orc_prefill(const void* q, const void* k, const void* v, int dtype, int64_t B,
                int64_t Hq, int64_t Hkv, int64_t S, int64_t D, int causal, double scale,
                double softcap, const int64_t* rows, int64_t nrows, double* y) {
  if (Hkv <= 0 || Hq % Hkv != 0) {
    return -1;
  }
  int64_t g = Hq / Hkv;
  int64_t total = B * Hq * S;
  int64_t count = rows ? nrows : total;
  orc_kv kv = {k, v, dtype, Hkv, S, D, D, 0, 0};
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)S);
  int* masked = (int*)malloc(sizeof(int) * (size_t)S);
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  for (int64_t r = 0; r < count; ++r) {
    int64_t row = rows ? rows[r] : r;
    int64_t i = row % S;
    int64_t h = (row / S) % Hq;
    int64_t b = row / (S * Hq);
    for (int64_t d = 0; d < D; ++d) {
      qr[d] = load_elem(q, ((b * Hq + h) * S + i) * D + d, dtype);
    }
    for (int64_t j = 0; j < S; ++j) {
      keys[j] = j;
      masked[j] = (causal && j > i) ? 1 : 0;
    }
    attend_row(&kv, b, h / g, qr, keys, masked, S, scale, softcap, NULL, NULL, y + r * D);
  }
  free(keys);
  free(masked);
  free(qr);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Paged causal decode ([PG] 16-token blocks through a table).               */
/* ------------------------------------------------------------------------ */

/* Pools [num_pages, Hkv, page_tokens, D]; token t of sequence b lives at
 * page block_table[b * max_pages + t / page_tokens], slot t % page_tokens.
 * The single new query of sequence b sits at position ctx_len[b] - 1 and
 * sees all ctx_len[b] tokens.  Gathers the sequence's keys into a contiguous
 * copy, then applies the dense formula.  Rows flattened (b, h). */
int orc_paged_decode(const void* q, const void* k_pool, const void* v_pool, int dtype,
                     const int32_t* block_table, const int32_t* ctx_len, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t D, int64_t page_tokens,
                     int64_t max_pages, double scale, const int64_t* rows, int64_t nrows,
                     double* y) {
  if (Hkv <= 0 || Hq % Hkv != 0) {
    return -1;
  }
  int64_t g = Hq / Hkv;
  int64_t total = B * Hq;
  int64_t count = rows ? nrows : total;
  size_t esz = dtype == ORC_F32 ? 4 : 2;
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  for (int64_t r = 0; r < count; ++r) {
    int64_t row = rows ? rows[r] : r;
    int64_t h = row % Hq;
    int64_t b = row / Hq;
    int64_t kvh = h / g;
    int64_t n = ctx_len[b];
    /* contiguous copy of this (b, kvh)'s keys/values, as [1, 1, n, D] */
    char* kc = (char*)malloc(esz * (size_t)(n * D > 0 ? n * D : 1));
    char* vc = (char*)malloc(esz * (size_t)(n * D > 0 ? n * D : 1));
    for (int64_t t = 0; t < n; ++t) {
      int64_t page = block_table[b * max_pages + t / page_tokens];
      int64_t slot = t % page_tokens;
      size_t src = (size_t)(((page * Hkv + kvh) * page_tokens + slot) * D) * esz;
      memcpy(kc + (size_t)(t * D) * esz, (const char*)k_pool + src, esz * (size_t)D);
      memcpy(vc + (size_t)(t * D) * esz, (const char*)v_pool + src, esz * (size_t)D);
    }
    for (int64_t d = 0; d < D; ++d) {
      qr[d] = load_elem(q, (b * Hq + h) * D + d, dtype);
    }
    orc_kv kv = {kc, vc, dtype, 1, n, D, D, 0, 0};
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int* masked = (int*)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    for (int64_t t = 0; t < n; ++t) {
      keys[t] = t;
    }
    attend_row(&kv, 0, 0, qr, keys, masked, n, scale, 0.0, NULL, NULL, y + r * D);
    free(keys);
    free(masked);
    free(kc);
    free(vc);
  }
  free(qr);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Ratio-4 index scoring and top-k selection.                                */
/*                                                                          */
/* [CSA-CPU] onnx-runtime-ep-cpu compressed_sparse_attention.rs:            */
/*   finalize_index_query, hadamard_bf16, fp4_roundtrip, select_ratio4_topk; */
/* [CSA] onnx-runtime-ep-cuda compressed_sparse_attention.rs:               */
/*   csa_ratio4_index_select (same steps on the device),                    */
/*   csa_ratio4_index_replicate (one shared set per index head).            */
/* OCP MX specification v1.0: E2M1 element encoding and the conversion of   */
/* a block of 32 scalars to an E8M0 scale plus elements.                    */
/*                                                                          */
/* The pages carry these steps out in binary32 arithmetic (plain f32 adds   */
/* and multiplies, bf16 rounding after the Hadamard transform), and the      */
/* results are integer decisions (FP4 codes, the order of scores), so this   */
/* section computes in float, in the pages' order, and does not widen to    */
/* double.  The build passes -ffp-contract=off: no step is fused.           */
/* ------------------------------------------------------------------------ */

#define ORC_SEL_TIE 1       /* two scores of the row compare equal           */
#define ORC_SEL_NONFINITE 2 /* a score is NaN or infinite                    */

/* OCP E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent field 0
 * is subnormal m * 0.5.  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_to_double(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int ex = (nibble >> 1) & 3;
  int m = nibble & 1;
  double v;
  if (ex == 0) {
    v = 0.5 * m;
  } else {
    v = ldexp(1.0 + 0.5 * m, ex - 1);
  }
  return sign ? -v : v;
}

/* Round a binary32 value to the nearest bfloat16 (ties to the even
 * neighbour), returned as binary32.  The two candidates are the value with
 * its low 16 bits cleared and the next bfloat16 away from zero. */
float orc_round_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) { /* inf stays inf, NaN a quiet NaN */
    if (u & 0x007fffffu) {
      u |= 0x00400000u;
    }
    u &= 0xffff0000u;
    memcpy(&x, &u, 4);
    return x;
  }
  uint32_t low = u & 0xffffu;
  uint32_t down = u & 0xffff0000u;
  int take_up = 0;
  if (low > 0x8000u) {
    take_up = 1;
  } else if (low == 0x8000u && ((down >> 16) & 1u)) {
    take_up = 1;
  }
  uint32_t r = take_up ? down + 0x10000u : down;
  float y;
  memcpy(&y, &r, 4);
  return y;
}

/* The nearest E2M1 magnitude code (0..7) to v >= 0, ties to the even code,
 * values beyond 6 saturating to 6 (code 7). */
static int orc_e2m1_nearest_code(double v) {
  int best = 0;
  double best_err = INFINITY;
  if (v > 6.0) {
    return 7;
  }
  for (int c = 0; c < 8; ++c) {
    double err = fabs(v - orc_e2m1_to_double((uint8_t)c));
    if (err < best_err || (err == best_err && (c % 2) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return best;
}

/* OCP MX conversion of one block of 32 binary32 scalars to FP4 E2M1 with an
 * E8M0 scale: X = 2^(floor(log2(amax)) - 2) (2 = the largest E2M1 exponent),
 * clamped to [2^-127, 2^127]; element i is the E2M1 value nearest x_i / X,
 * ties to even, saturating at +-6.  An all-zero block takes scale byte 0; a
 * block holding inf or NaN takes the NaN scale byte 0xFF and zero codes.
 * packed[j] holds element 2j in its low nibble and 2j+1 in its high nibble. */
void orc_fp4_quantize_block(const float* x, uint8_t* scale_byte, uint8_t* packed) {
  double amax = 0.0;
  int finite = 1;
  for (int i = 0; i < 32; ++i) {
    double a = fabs((double)x[i]);
    if (!isfinite(a)) {
      finite = 0;
    }
    if (a > amax) {
      amax = a;
    }
  }
  for (int j = 0; j < 16; ++j) {
    packed[j] = 0;
  }
  if (!finite) {
    *scale_byte = 0xff;
    return;
  }
  if (amax == 0.0) {
    *scale_byte = 0;
    return;
  }
  int k;
  frexp(amax, &k); /* amax = f * 2^k, f in [0.5, 1): floor(log2 amax) = k - 1 */
  int e = (k - 1) - 2;
  if (e < -127) {
    e = -127;
  }
  if (e > 127) {
    e = 127;
  }
  *scale_byte = (uint8_t)(e + 127);
  for (int i = 0; i < 32; ++i) {
    double v = ldexp((double)x[i], -e);
    int code = orc_e2m1_nearest_code(fabs(v));
    if (v < 0.0 && code != 0) {
      code |= 8;
    }
    packed[i / 2] |= (uint8_t)((i % 2) ? (code << 4) : code);
  }
}

/* Element i of an FP4 block: e2m1(code) * 2^(scale - 127), NaN for 0xFF. */
float orc_fp4_element(uint8_t scale_byte, const uint8_t* packed, int i) {
  uint8_t nib = (uint8_t)((i % 2) ? (packed[i / 2] >> 4) : (packed[i / 2] & 0xf));
  if (scale_byte == 0xff) {
    return NAN;
  }
  return (float)ldexp(orc_e2m1_to_double(nib), (int)scale_byte - 127);
}

/* [CSA-CPU] hadamard_bf16: the unnormalised Walsh-Hadamard transform by
 * butterflies (span 1, 2, 4, ...: a + b, a - b in binary32), then every value
 * times 1/sqrt(n) (binary32) and rounded to bfloat16.  n a power of two. */
void orc_hadamard_bf16(float* v, int64_t n) {
  for (int64_t span = 1; span < n; span *= 2) {
    for (int64_t start = 0; start < n; start += 2 * span) {
      for (int64_t off = 0; off < span; ++off) {
        float a = v[start + off];
        float b = v[start + off + span];
        v[start + off] = a + b;
        v[start + off + span] = a - b;
      }
    }
  }
  float scale = 1.0f / sqrtf((float)n);
  for (int64_t i = 0; i < n; ++i) {
    float p = v[i] * scale;
    v[i] = orc_round_bf16(p);
  }
}

/* [CSA-CPU] finalize_index_query: bfloat16 rounding of the query head, then
 * (RoPE of its last components is applied by the caller before this step)
 * the Hadamard transform and an FP4 round trip per block of 32 (quantize,
 * then dequantize in place).  out may equal src. */
void orc_index_query_finalize(const float* src, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    out[i] = orc_round_bf16(src[i]);
  }
  orc_hadamard_bf16(out, n);
  for (int64_t blk = 0; blk < n / 32; ++blk) {
    uint8_t sb, packed[16];
    orc_fp4_quantize_block(out + 32 * blk, &sb, packed);
    for (int i = 0; i < 32; ++i) {
      out[32 * blk + i] = orc_fp4_element(sb, packed, i);
    }
  }
}

/* Rust's f32::total_cmp as a signed integer key: for negative values every
 * bit but the sign is flipped, so the signed order of the keys is the total
 * order (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN). */
static int32_t orc_total_key(float f) {
  int32_t k;
  memcpy(&k, &f, 4);
  if (k < 0) {
    k ^= 0x7fffffff;
  }
  return k;
}

typedef struct {
  int32_t record;
  float score;
} orc_scored;

/* Higher score first (total order), then the lower record. */
static int orc_rank_cmp(const void* pa, const void* pb) {
  const orc_scored* a = (const orc_scored*)pa;
  const orc_scored* b = (const orc_scored*)pb;
  int32_t ka = orc_total_key(a->score), kb = orc_total_key(b->score);
  if (ka != kb) {
    return ka > kb ? -1 : 1;
  }
  return (a->record > b->record) - (a->record < b->record);
}

static int orc_int_cmp(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

typedef struct {
  const float* query;    /* [B, S, IH, ID] */
  const float* weight;   /* [B, S, IH] */
  const uint8_t* keys;   /* [B, R, key_stride]: ID/32 blocks of [scale, 16 packed bytes] */
  int64_t B, S, IH, ID, R, topk, key_stride;
  int64_t query_start;           /* position of query s is query_start + s ... */
  const int64_t* query_start_b;  /* ... or query_start_b[b] + s when given */
  int64_t out_heads;             /* copies of the set: selected [B, out_heads, S, topk] */
  int ascending;                 /* 0: score order; 1: ascending record order */
} orc_select_args;

/* [CSA-CPU] select_ratio4_topk.  For row (b, s) at position p, the causal
 * records are r < min(R, (p + 1) / 4).  Each record's score is
 *   sum over heads h (ascending) of relu(q_h . k_r) * w_h * c,
 *   c = (1/sqrt(ID)) / sqrt(IH), q_h the finalized query head,
 * the dot product summed in ascending dimension order, every operation in
 * binary32 and unfused.  The records are ranked by score (higher first,
 * Rust total_cmp) and then by record index; the first topk fill the row,
 * -1 the rest.  Two equal scores in a row set SEL_TIE (the pages refuse such
 * input; the ranking still orders them by record), a non-finite score sets
 * SEL_NONFINITE.  scores (nullable) receives [B, S, R] (0 past the causal
 * limit).  Returns 0, or -1 on a bad shape. */
int orc_index_select(const orc_select_args* a, int32_t* selected, uint8_t* status,
                     uint32_t* err, float* scores) {
  if (a->ID <= 0 || a->ID % 32 != 0 || (a->ID & (a->ID - 1)) != 0 || a->IH <= 0 ||
      a->topk <= 0 || a->key_stride < a->ID / 32 * 17 || a->out_heads <= 0) {
    return -1;
  }
  uint32_t acc = 0;
  float* q = (float*)malloc(sizeof(float) * (size_t)(a->IH * a->ID));
  float* k = (float*)malloc(sizeof(float) * (size_t)a->ID);
  orc_scored* rank = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)(a->R > 0 ? a->R : 1));
  int32_t* row = (int32_t*)malloc(sizeof(int32_t) * (size_t)a->topk);
  float c = 1.0f / sqrtf((float)a->ID);
  c = c / sqrtf((float)a->IH);
  for (int64_t b = 0; b < a->B; ++b) {
    for (int64_t s = 0; s < a->S; ++s) {
      int64_t pos = (a->query_start_b ? a->query_start_b[b] : a->query_start) + s;
      int64_t limit = pos >= 0 ? (pos + 1) / 4 : 0;
      if (limit > a->R) {
        limit = a->R;
      }
      for (int64_t h = 0; h < a->IH; ++h) {
        const float* src = a->query + ((b * a->S + s) * a->IH + h) * a->ID;
        orc_index_query_finalize(src, a->ID, q + h * a->ID);
      }
      const float* w = a->weight + (b * a->S + s) * a->IH;
      int code = 0;
      for (int64_t r = 0; r < limit; ++r) {
        const uint8_t* rec = a->keys + (b * a->R + r) * a->key_stride;
        for (int64_t d = 0; d < a->ID; ++d) {
          const uint8_t* blk = rec + (d / 32) * 17;
          k[d] = orc_fp4_element(blk[0], blk + 1, (int)(d % 32));
        }
        float score = 0.0f;
        for (int64_t h = 0; h < a->IH; ++h) {
          float dot = 0.0f;
          for (int64_t d = 0; d < a->ID; ++d) {
            float p = q[h * a->ID + d] * k[d];
            dot = dot + p;
          }
          float relu = fmaxf(dot, 0.0f);
          float t = relu * w[h];
          t = t * c;
          score = score + t;
        }
        if (!isfinite(score)) {
          code |= ORC_SEL_NONFINITE;
        }
        rank[r].record = (int32_t)r;
        rank[r].score = score;
      }
      if (scores) {
        for (int64_t r = 0; r < a->R; ++r) {
          scores[(b * a->S + s) * a->R + r] = r < limit ? rank[r].score : 0.0f;
        }
      }
      /* equal scores: sort a copy of the scores, compare neighbours with == */
      {
        float* sorted = (float*)malloc(sizeof(float) * (size_t)(limit > 0 ? limit : 1));
        orc_scored* tmp = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)(limit > 0 ? limit : 1));
        memcpy(tmp, rank, sizeof(orc_scored) * (size_t)limit);
        qsort(tmp, (size_t)limit, sizeof(orc_scored), orc_rank_cmp);
        for (int64_t r = 0; r < limit; ++r) {
          sorted[r] = tmp[r].score;
        }
        for (int64_t r = 1; r < limit; ++r) {
          if (sorted[r] == sorted[r - 1]) {
            code |= ORC_SEL_TIE;
          }
        }
        free(sorted);
        free(tmp);
      }
      qsort(rank, (size_t)limit, sizeof(orc_scored), orc_rank_cmp);
      int64_t n = limit < a->topk ? limit : a->topk;
      for (int64_t j = 0; j < a->topk; ++j) {
        row[j] = j < n ? rank[j].record : -1;
      }
      if (a->ascending) {
        qsort(row, (size_t)n, sizeof(int32_t), orc_int_cmp);
      }
      for (int64_t o = 0; o < a->out_heads; ++o) {
        memcpy(selected + ((b * a->out_heads + o) * a->S + s) * a->topk, row,
               sizeof(int32_t) * (size_t)a->topk);
      }
      if (status) {
        status[b * a->S + s] = (uint8_t)code;
      }
      acc |= (uint32_t)code;
    }
  }
  free(q);
  free(k);
  free(rank);
  free(row);
  if (err) {
    *err = acc;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Compressed sparse attention, ratio 4, in the pages' own form.             */
/*                                                                          */
/* [CSA-CPU] ratio4_attention and its call in execute_ratio4; [CSA]         */
/* csa_ratio4_sink_attention.  A separate dense window store (current_kv,   */
/* one latent head, K = V) of the most recent tokens and the selected       */
/* compressed records (hybrid FP8, K = V = the decoded record) are the      */
/* candidates; an optional additive bias is keyed by the candidate slot; a  */
/* per-head sink logit joins the softmax denominator.                       */
/* ------------------------------------------------------------------------ */

typedef struct {
  const void* query;      /* [B, S, H, D] f32 or bf16 (q_dtype) */
  int q_dtype;
  const void* window;     /* [B, L, D] f32 or bf16 (w_dtype): current_kv */
  int w_dtype;
  const uint8_t* records; /* [B, R, record_bytes] hybrid FP8 records */
  const int32_t* selected;/* [B, S, topk] record indices, -1 padded */
  const double* sink;     /* nullable [H] */
  const float* bias;      /* nullable: rank bias_rank, broadcast against [B, H, S, C] */
  int64_t bias_rank;
  int64_t bias_dims[4];
  int64_t B, S, H, D, L, R, topk, record_bytes, n_rope;
  int64_t total;          /* tokens so far (the current ones included) */
  double scale;           /* 0: 1/sqrt(D) */
} orc_csa_args;

/* Returns 0, -1 on a bad shape; *bad_record = 1 when a selected entry is at
 * or past the valid records (such a slot is skipped, as the device kernel of
 * the pages does; their CPU reference refuses the input).  y [B, S, H, D]. */
int orc_csa_ratio4_attention(const orc_csa_args* a, double* y, int* bad_record) {
  int64_t query_start = a->total - a->S;
  int64_t base = a->total - a->L; /* position of current_kv row 0 */
  int64_t valid_records = a->total / 4;
  if (valid_records > a->R) {
    valid_records = a->R;
  }
  int64_t dense = 128;
  if (query_start == 0) {
    dense = a->L < 128 ? a->L : 128;
  }
  int64_t C = dense + a->topk;
  if (a->bias) {
    int64_t target[4] = {a->B, a->H, a->S, C};
    if (a->bias_rank < 0 || a->bias_rank > 4) {
      return -1;
    }
    for (int64_t r = 0; r < a->bias_rank; ++r) {
      int64_t t = target[4 - a->bias_rank + r];
      if (a->bias_dims[r] != 1 && a->bias_dims[r] != t) {
        return -1;
      }
    }
  }
  double scale = a->scale != 0.0 ? a->scale : 1.0 / sqrt((double)a->D);
  double* s = (double*)malloc(sizeof(double) * (size_t)C);
  double* q = (double*)malloc(sizeof(double) * (size_t)a->D);
  double* rows = (double*)malloc(sizeof(double) * (size_t)(C * a->D));
  int* valid = (int*)malloc(sizeof(int) * (size_t)C);
  *bad_record = 0;
  for (int64_t b = 0; b < a->B; ++b) {
    for (int64_t si = 0; si < a->S; ++si) {
      int64_t pos = query_start + si;
      int64_t wstart = pos + 1 - 128;
      if (wstart < 0) {
        wstart = 0;
      }
      int64_t dense_start = base > wstart ? base : wstart;
      /* the candidates' rows, shared by every head */
      for (int64_t c = 0; c < C; ++c) {
        valid[c] = 0;
        double* row = rows + c * a->D;
        if (c < dense) {
          int64_t absolute = dense_start + c;
          int64_t rel = absolute - base;
          if (absolute > pos || rel < 0 || rel >= a->L) {
            continue;
          }
          for (int64_t d = 0; d < a->D; ++d) {
            row[d] = load_elem(a->window, (b * a->L + rel) * a->D + d, a->w_dtype);
          }
          valid[c] = 1;
        } else {
          int32_t rec = a->selected[(b * a->S + si) * a->topk + (c - dense)];
          if (rec < 0) {
            continue;
          }
          if (rec >= valid_records) {
            *bad_record = 1;
            continue;
          }
          orc_decode_fp8_record(a->records + (b * a->R + rec) * a->record_bytes,
                                a->D - a->n_rope, a->n_rope, row);
          valid[c] = 1;
        }
      }
      for (int64_t h = 0; h < a->H; ++h) {
        double* out = y + ((b * a->S + si) * a->H + h) * a->D;
        for (int64_t d = 0; d < a->D; ++d) {
          q[d] = load_elem(a->query, ((b * a->S + si) * a->H + h) * a->D + d, a->q_dtype);
          out[d] = 0.0;
        }
        double M = -INFINITY;
        for (int64_t c = 0; c < C; ++c) {
          s[c] = -INFINITY;
          if (!valid[c]) {
            continue;
          }
          double dot = 0.0;
          for (int64_t d = 0; d < a->D; ++d) {
            dot += q[d] * rows[c * a->D + d];
          }
          double sc = dot * scale;
          if (a->bias) {
            sc += orc_bias_at(a->bias, a->bias_rank, a->bias_dims, b, h, si, c);
          }
          s[c] = sc;
          if (sc > M) {
            M = sc;
          }
        }
        if (M == -INFINITY) {
          continue; /* no candidate: the row stays 0 */
        }
        double den = 0.0;
        for (int64_t c = 0; c < C; ++c) {
          if (s[c] != -INFINITY) {
            den += exp(s[c] - M);
          }
        }
        if (a->sink) {
          den += exp(a->sink[h] - M);
        }
        for (int64_t c = 0; c < C; ++c) {
          if (s[c] == -INFINITY) {
            continue;
          }
          double p = exp(s[c] - M) / den;
          for (int64_t d = 0; d < a->D; ++d) {
            out[d] += p * rows[c * a->D + d];
          }
        }
      }
    }
  }
  free(s);
  free(q);
  free(rows);
  free(valid);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* CSA compression: ratio 128 and ratio 4 (attention records, index keys).  */
/*                                                                          */
/* [CSA-CPU] compress_ratio4_stream, pool_ratio4_record,                    */
/* pool_ratio128_record, finalize_attention_record, finalize_index_record,  */
/* apply_compressed_rope; [CSA] csa_ratio128_compress,                      */
/* csa_ratio4_main_compress, csa_ratio4_index_compress.  Binary32           */
/* arithmetic, one rounding per operation, in the pages' order (the pages   */
/* fix the record bytes, so the oracle reproduces their precision rather    */
/* than widening to double).  Each transcendental value (the pool weight,   */
/* the RoPE base frequency, sine and cosine) is the binary32 rounding of a  */
/* double evaluation, the device page's own form for the pool weight.       */
/* ------------------------------------------------------------------------ */

#define ORC_COMPRESS_ATTN 0  /* hybrid FP8 attention record */
#define ORC_COMPRESS_INDEX 1 /* FP4 index key (Hadamard first) */

/* e^t rounded to binary32, t = score - max (<= 0): [CSA] ratio-4 pooling. */
float orc_pool_weight(float t) {
  return (float)exp((double)t);
}

/* Compressed RoPE rotation at `position` for n_rope/2 pairs ([CSA-CPU]
 * apply_compressed_rope): base 160000, factor 16, ramp over pairs 15..25. */
void orc_rope_rotation(int64_t position, int64_t n_rope, float* cs, float* sn) {
  float p = (float)position;
  for (int64_t pair = 0; pair < n_rope / 2; ++pair) {
    float ramp = ((float)pair - 15.0f) / 10.0f;
    if (ramp < 0.0f) {
      ramp = 0.0f;
    }
    if (ramp > 1.0f) {
      ramp = 1.0f;
    }
    float ex = -((float)(2 * pair)) / (float)n_rope;
    float base = (float)pow(160000.0, (double)ex);
    float t1 = base * (1.0f - ramp);
    float t2 = (base / 16.0f) * ramp;
    float freq = t1 + t2;
    float angle = p * freq;
    cs[pair] = (float)cos((double)angle);
    sn[pair] = (float)sin((double)angle);
  }
}

/* E4M3FN code nearest to v (|v| <= 448), ties to the even code, the sign of
 * v kept (so -0 and negative values rounding to zero give 0x80). */
static uint8_t orc_e4m3fn_nearest(double v) {
  double mag = fabs(v);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c < 0x7f; ++c) {
    double err = fabs(mag - orc_e4m3fn_to_double((uint8_t)c));
    if (err < best_err || (err == best_err && (c % 2) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(signbit(v) ? (0x80 | best) : best);
}

/* One FP8 block: out[0] = E8M0 byte of the smallest e with amax / 2^e <= 448
 * (e = 0 for an all-zero block, clamped to [-127, 127]); out[1 + i] = the
 * nearest E4M3FN code of x_i / 2^e.  The values must be finite. */
void orc_fp8_quantize_block(const float* x, uint8_t* out) {
  double amax = 0.0;
  for (int i = 0; i < 64; ++i) {
    double m = fabs((double)x[i]);
    if (m > amax) {
      amax = m;
    }
  }
  int e = 0;
  if (amax > 0.0) {
    int k;
    double f = frexp(amax, &k); /* amax = f * 2^k, f in [0.5, 1); 448 = 0.875 * 2^9 */
    e = k - 9 + (f > 0.875 ? 1 : 0);
    if (e < -127) {
      e = -127;
    }
    if (e > 127) {
      e = 127;
    }
  }
  out[0] = (uint8_t)(e + 127);
  for (int i = 0; i < 64; ++i) {
    out[1 + i] = orc_e4m3fn_nearest(ldexp((double)x[i], -e));
  }
}

static int orc_all_finite(const float* v, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    if (!isfinite(v[i])) {
      return 0;
    }
  }
  return 1;
}

/* Softmax pooling of one dimension over n candidates ([CSA-CPU]
 * pool_ratio4_record / pool_ratio128_record): the maximum score, then in
 * candidate order every score that is not -inf adds its weight to the
 * denominator and weight * value to the numerator.  Returns 0 when the
 * maximum is not finite or the sums are not usable. */
static int orc_pool_dim(const float* value, const float* score, int64_t n, float* out) {
  float m = -INFINITY;
  for (int64_t c = 0; c < n; ++c) {
    m = fmaxf(m, score[c]);
  }
  if (!isfinite(m)) {
    return 0;
  }
  float num = 0.0f, den = 0.0f;
  for (int64_t c = 0; c < n; ++c) {
    if (score[c] == -INFINITY) {
      continue;
    }
    float w = orc_pool_weight(score[c] - m);
    num = num + w * value[c];
    den = den + w;
  }
  if (den == 0.0f || !isfinite(den) || !isfinite(num)) {
    return 0;
  }
  *out = num / den;
  return 1;
}

/* The pooled candidates of one record, exported for the tests: value and
 * score are [n, D]; out [D].  Returns 0 when a dimension fails to pool. */
int orc_pool_candidates(const float* value, const float* score, int64_t n, int64_t D,
                        float* out) {
  float* v = (float*)malloc(sizeof(float) * (size_t)n);
  float* s = (float*)malloc(sizeof(float) * (size_t)n);
  int ok = 1;
  for (int64_t d = 0; d < D; ++d) {
    for (int64_t c = 0; c < n; ++c) {
      v[c] = value[c * D + d];
      s[c] = score[c * D + d];
    }
    if (!orc_pool_dim(v, s, n, out + d)) {
      ok = 0;
      out[d] = 0.0f;
    }
  }
  free(v);
  free(s);
  return ok;
}

/* Finalize one pooled record ([CSA-CPU] finalize_attention_record /
 * finalize_index_record): bfloat16 rounding; RMSNorm (binary32 square sum
 * in dimension order, 1 / sqrt(sum / D + 1e-6)) times the learned scale,
 * bfloat16; the compressed RoPE of the last n_rope dimensions at
 * block_start, bfloat16 per component.  Attention records then quantize the
 * first D - n_rope dimensions per block of 64 to FP8 and store the RoPE
 * tail as little-endian bfloat16; index keys take the Hadamard transform and
 * quantize per block of 32 to FP4.  `rec` holds the pooled values on entry
 * and the logical (dequantized) record on return; `bytes` gets the stored
 * record.  Returns 0 (and zeroes both) when a value is not finite. */
int orc_finalize_record(float* rec, const float* norm, int64_t D, int64_t n_rope, int kind,
                        int64_t block_start, uint8_t* bytes) {
  int64_t width = kind == ORC_COMPRESS_ATTN ? ((D - n_rope) / 64) * 65 + 2 * n_rope
                                            : (D / 32) * 17;
  for (int64_t d = 0; d < D; ++d) {
    rec[d] = orc_round_bf16(rec[d]);
  }
  float sum = 0.0f;
  for (int64_t d = 0; d < D; ++d) {
    sum = sum + rec[d] * rec[d];
  }
  int ok = isfinite(sum) && orc_all_finite(rec, D);
  if (ok) {
    float inv = 1.0f / sqrtf(sum / (float)D + 1.0e-6f);
    for (int64_t d = 0; d < D; ++d) {
      rec[d] = orc_round_bf16((rec[d] * inv) * norm[d]);
    }
    float* cs = (float*)malloc(sizeof(float) * (size_t)(n_rope / 2 + 1));
    float* sn = (float*)malloc(sizeof(float) * (size_t)(n_rope / 2 + 1));
    orc_rope_rotation(block_start, n_rope, cs, sn);
    for (int64_t pair = 0; pair < n_rope / 2; ++pair) {
      int64_t d = D - n_rope + 2 * pair;
      float re = rec[d], im = rec[d + 1];
      rec[d] = orc_round_bf16(re * cs[pair] - im * sn[pair]);
      rec[d + 1] = orc_round_bf16(re * sn[pair] + im * cs[pair]);
    }
    free(cs);
    free(sn);
    if (kind == ORC_COMPRESS_INDEX) {
      orc_hadamard_bf16(rec, D);
    }
    ok = orc_all_finite(rec, D);
  }
  if (!ok) {
    for (int64_t d = 0; d < D; ++d) {
      rec[d] = 0.0f;
    }
    memset(bytes, 0, (size_t)width);
    return 0;
  }
  if (kind == ORC_COMPRESS_ATTN) {
    int64_t nb = (D - n_rope) / 64;
    for (int64_t blk = 0; blk < nb; ++blk) {
      uint8_t* p = bytes + blk * 65;
      orc_fp8_quantize_block(rec + blk * 64, p);
      double s = orc_e8m0_to_double(p[0]);
      for (int64_t i = 0; i < 64; ++i) {
        rec[blk * 64 + i] = (float)(orc_e4m3fn_to_double(p[1 + i]) * s);
      }
    }
    uint8_t* tail = bytes + nb * 65;
    for (int64_t r = 0; r < n_rope; ++r) {
      float v = rec[D - n_rope + r];
      uint32_t u;
      memcpy(&u, &v, 4);
      tail[2 * r] = (uint8_t)((u >> 16) & 0xff);
      tail[2 * r + 1] = (uint8_t)(u >> 24);
    }
  } else {
    for (int64_t blk = 0; blk < D / 32; ++blk) {
      uint8_t* p = bytes + blk * 17;
      orc_fp4_quantize_block(rec + blk * 32, p, p + 1);
      for (int i = 0; i < 32; ++i) {
        rec[blk * 32 + i] = orc_fp4_element(p[0], p + 1, i);
      }
    }
  }
  return 1;
}

typedef struct {
  const float* kv;   /* [B, S, W] the compressor's value source, W = D (ratio 128) or 2D */
  const float* gate; /* [B, S, W] the compressor's score source */
  const float* ape;  /* [ratio, W] positional score bias, by position within the block */
  const float* norm; /* [D] RMSNorm scale */
  float* carry;      /* [B, slots, 2, W], slots = 128 or 8; channel 0 value, 1 score */
  uint8_t* records;  /* nullable [B, rows, record_stride] stored records */
  float* logical;    /* nullable [B, rows, D] the dequantized records */
  int64_t B, S, D, n_rope, ratio, kind, rows, record_stride, total;
} orc_compress_args;

/* The compression stream ([CSA-CPU] compress_ratio4_stream and the ratio-128
 * loop; [CSA] csa_ratio*_compress), token by token: the token's value and
 * gate + ape fill its carry slot (ratio 128: slot pos % 128; ratio 4: the
 * current-window slot 4 + pos % 4); at the end of every block of `ratio`
 * tokens the carry is pooled into one record (ratio 4: candidates 0..3 are
 * the previous block's slots on the first D source dimensions, 4..7 the
 * current block's on the last D), finalized at block_start = pos + 1 -
 * ratio and stored as record pos / ratio; then the carry is cleared (ratio
 * 128) or the current window moves into the previous one and is cleared
 * (ratio 4).  A stream starting at position 0 starts from a cleared carry.
 * A record that fails to pool or finalize is stored as zeros and counted in
 * *invalid.  Returns -1 on a bad shape. */
int orc_csa_compress(const orc_compress_args* a, int64_t* invalid) {
  int64_t R = a->ratio, D = a->D;
  if (R != 4 && R != 128) {
    return -1;
  }
  if (a->kind == ORC_COMPRESS_INDEX && R != 4) {
    return -1;
  }
  if (a->n_rope < 0 || a->n_rope > D || a->n_rope % 2) {
    return -1;
  }
  if (a->kind == ORC_COMPRESS_ATTN && (D - a->n_rope) % 64) {
    return -1;
  }
  if (a->kind == ORC_COMPRESS_INDEX && (D % 32 || (D & (D - 1)))) {
    return -1;
  }
  int64_t start = a->total - a->S;
  if (start < 0 || a->S < 0 || a->total / R > a->rows) {
    return -1;
  }
  int64_t width = a->kind == ORC_COMPRESS_ATTN ? ((D - a->n_rope) / 64) * 65 + 2 * a->n_rope
                                               : (D / 32) * 17;
  if (a->records && a->record_stride < width) {
    return -1;
  }
  int64_t slots = R == 128 ? 128 : 8;
  int64_t W = R == 4 ? 2 * D : D;
  int64_t ncand = R == 128 ? 128 : 8;
  float* rec = (float*)malloc(sizeof(float) * (size_t)D);
  float* cv = (float*)malloc(sizeof(float) * (size_t)ncand);
  float* cscore = (float*)malloc(sizeof(float) * (size_t)ncand);
  uint8_t* bytes = (uint8_t*)malloc((size_t)width);
  *invalid = 0;
  for (int64_t b = 0; b < a->B; ++b) {
    float* cy = a->carry + b * slots * 2 * W;
    if (start == 0) {
      for (int64_t sl = 0; sl < slots; ++sl) {
        for (int64_t d = 0; d < W; ++d) {
          cy[(sl * 2) * W + d] = 0.0f;
          cy[(sl * 2 + 1) * W + d] = -INFINITY;
        }
      }
    }
    for (int64_t s = 0; s < a->S; ++s) {
      int64_t pos = start + s;
      int64_t phase = pos % R;
      int64_t slot = R == 4 ? 4 + phase : phase;
      const float* kv = a->kv + (b * a->S + s) * W;
      const float* gate = a->gate + (b * a->S + s) * W;
      for (int64_t d = 0; d < W; ++d) {
        cy[(slot * 2) * W + d] = kv[d];
        cy[(slot * 2 + 1) * W + d] = gate[d] + a->ape[phase * W + d];
      }
      if ((pos + 1) % R != 0) {
        continue;
      }
      int ok = 1;
      for (int64_t d = 0; d < D; ++d) {
        for (int64_t c = 0; c < ncand; ++c) {
          int64_t sd = (R == 4 && c >= 4) ? D + d : d;
          cv[c] = cy[(c * 2) * W + sd];
          cscore[c] = cy[(c * 2 + 1) * W + sd];
        }
        if (!orc_pool_dim(cv, cscore, ncand, rec + d)) {
          ok = 0;
          rec[d] = 0.0f;
        }
      }
      if (ok) {
        ok = orc_finalize_record(rec, a->norm, D, a->n_rope, (int)a->kind, pos + 1 - R, bytes);
      } else {
        memset(rec, 0, sizeof(float) * (size_t)D);
        memset(bytes, 0, (size_t)width);
      }
      if (!ok) {
        *invalid += 1;
      }
      int64_t out = pos / R;
      if (a->records) {
        memcpy(a->records + (b * a->rows + out) * a->record_stride, bytes, (size_t)width);
      }
      if (a->logical) {
        memcpy(a->logical + (b * a->rows + out) * D, rec, sizeof(float) * (size_t)D);
      }
      if (R == 128) {
        for (int64_t sl = 0; sl < 128; ++sl) {
          for (int64_t d = 0; d < W; ++d) {
            cy[(sl * 2) * W + d] = 0.0f;
            cy[(sl * 2 + 1) * W + d] = -INFINITY;
          }
        }
      } else {
        for (int64_t prev = 0; prev < 4; ++prev) {
          for (int64_t ch = 0; ch < 2; ++ch) {
            for (int64_t d = 0; d < W; ++d) {
              cy[(prev * 2 + ch) * W + d] = cy[((4 + prev) * 2 + ch) * W + d];
              cy[((4 + prev) * 2 + ch) * W + d] = ch == 0 ? 0.0f : -INFINITY;
            }
          }
        }
      }
    }
  }
  free(rec);
  free(cv);
  free(cscore);
  free(bytes);
  return 0;
}
