/*
 * sa.h -- C ABI of the GB300 KV-cache attention library (libsa.so).
 *
 * Eight operations, all computed on the GPU on the caller's stream:
 *
 *   validate_indices     index-row validation with a device error word
 *   build_present_kv     present K/V = past ++ current (concat or in-place append)
 *   sparse_attn_decode   selected-token attention (dense or FP8 hybrid cache)
 *   attn_prefill         dense (causal) prefill with softcap, present K/V out
 *   paged_attn_decode    causal decode over a 16-token page table
 *   sparse_index_select  ratio-4 index scoring + top-k (produces selected indices)
 *   csa_ratio4_attention compressed sparse attention: window store + records + sink
 *   csa_*_compress       the compression stages that produce the CSA records
 *                        (ratio 128, ratio-4 attention records, ratio-4 index keys)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *    library never allocates, frees or synchronises; scratch comes from a
 *    caller-provided workspace whose size is given by the matching
 *    *_workspace() query.  Tensors are dense and row-major in the stated
 *    shape (no strides other than the stated capacity strides).
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  All work is enqueued on it; the calls return before it runs.
 *  - Host-side argument errors return a negative status before anything is
 *    enqueued.  Data-dependent problems (malformed index rows, out-of-range
 *    page table entries or write positions) never fail the call: they OR bits
 *    into a caller-zeroed device word `err_word` (read it after your own
 *    synchronisation), and the kernels keep every load in bounds.
 *  - The calls are stateless and thread-safe.  No kernel spins or traps.
 *
 * Sources of the semantics (page title, section):
 *  [IS]  onnx-runtime-ep-cuda src/kernels/index_share.rs (IndexShare):
 *        module docs, validate_indices, build_present, index_share_row.
 *  [SA]  onnx-runtime-ep-cuda src/kernels/standard_attention.rs (ONNX
 *        Attention): module docs "Semantics", build_kv, attention_row,
 *        attention_split / attention_combine (FlashDecoding split-KV).
 *  [CSA] onnx-runtime-ep-cpu src/kernels/compressed_sparse_attention.rs:
 *        CacheFormat (hybrid FP8 record), dequantize_cache; onnx-runtime-ep-cuda
 *        compressed_sparse_attention.rs, csa_ratio128_sink_attention.
 *  [PG]  ferrum-kernels vnext_ops/transformer/causal_attention.rs: paged KV
 *        blocks of 16 tokens addressed through a table.
 *  [CSA-CPU] onnx-runtime-ep-cpu compressed_sparse_attention.rs: the ratio-4
 *        index stream (finalize_index_query, select_ratio4_topk) and the
 *        compression stream (compress_ratio4_stream, pool_ratio4_record,
 *        pool_ratio128_record, finalize_attention_record,
 *        finalize_index_record, apply_compressed_rope).
 */
#ifndef SA_H
#define SA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ------------------------------------ */
#define SA_OK 0
#define SA_ERR_NULL (-1)        /* a required pointer is NULL                 */
#define SA_ERR_SHAPE (-2)       /* a size is non-positive or inconsistent     */
#define SA_ERR_DTYPE (-3)       /* unsupported dtype or dtype combination     */
#define SA_ERR_ALIGN (-4)       /* a pointer is not 16-byte aligned           */
#define SA_ERR_WORKSPACE (-5)   /* workspace missing or too small             */
#define SA_ERR_OVERLAP (-6)     /* an output overlaps an input illegally      */
#define SA_ERR_UNSUPPORTED (-7) /* valid request this build does not serve    */
#define SA_ERR_LAUNCH (-8)      /* the CUDA runtime refused a launch          */
#define SA_ERR_SCRATCH_LIMIT (-9) /* sparse_attn_decode_noalloc: scratch needed
                                     exceeds SA_NOALLOC_SCRATCH_BYTES          */

/* ---- storage dtypes --------------------------------------------------- */
#define SA_F32 0
#define SA_F16 1
#define SA_BF16 2
#define SA_FP8_E4M3_B64 3 /* hybrid record: blocks of [E8M0, 64 x E4M3FN] + bf16 tail */

/* ---- index-row status codes (row_status bytes; OR-ed into err_word) --- */
#define SA_IDX_BELOW_SENTINEL 1  /* a value below -1                          */
#define SA_IDX_AFTER_PADDING 2   /* a non -1 value after a -1                 */
#define SA_IDX_OUT_OF_RANGE 4    /* a value >= the row's bound                */
#define SA_IDX_NOT_INCREASING 8  /* a value smaller than its predecessor      */
#define SA_IDX_DUPLICATE 16      /* a value equal to its predecessor          */
#define SA_IDX_ALL_PADDING 32    /* the row holds only -1                     */
/* other err_word bits */
#define SA_ERRBIT_WRITE_POS 64   /* build_present_kv: write_pos[b] out of range */
#define SA_ERRBIT_PAGE 128       /* paged: ctx_len or block-table entry invalid */
#define SA_ERRBIT_TIMEOUT 256    /* a kernel's bounded wait for a copy ran out  */
#define SA_ERRBIT_RECORD 2048    /* csa_ratio4_attention: a selected record at or
                                    past the valid records (skipped)             */
#define SA_ERRBIT_COMPRESS 4096  /* csa_*_compress: a record met a non-finite
                                    value and was stored as zeros                */

/* ---- sa_sparse_params.options bits ------------------------------------- */
#define SA_OPT_ROW_COPIES 1u     /* dense f16/bf16 caches: fetch each K/V row with
                                    its own bulk copy instead of TMA tensor maps */
#define SA_OPT_FP8_WARP_MMA 2u   /* FP8 records: the warp-level MMA kernel (32-head
                                    blocks) for every head count */

/* Human-readable name of a status code (static string). */
const char* sa_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int sa_version(void);

/*
 * sa_set_kernel_events -- measurement hook (no counterpart on the pages).
 *
 * before, after: cudaEvent_t handles (created by the caller, with timing
 * enabled), or both NULL to turn the hook off.  While set, every call made
 * from this host thread records `before` on its stream immediately before it
 * launches its dominant kernel (the gather kernel of a decode, the tensor-core
 * attention kernel of an FP8 decode, the prefill kernel) and `after`
 * immediately after it, so that the events bracket that one kernel.  The
 * handles are not owned; the caller keeps them alive while the hook is set.
 * Recording between two kernels removes their launch overlap, so timings of
 * whole calls are taken with the hook off.  Under stream capture the records
 * become event-record nodes of the graph (cudaEventRecordExternal), so a
 * replayed graph brackets the kernel the same way.
 * Returns SA_OK, or SA_ERR_NULL if exactly one of the two is NULL.
 */
int sa_set_kernel_events(void* before, void* after);

/*
 * sa_graph_kernel_count -- measurement hook (no counterpart on the pages): the
 * number of kernel nodes in a CUDA graph (a cudaGraph_t, not owned), e.g. one
 * library call captured from a stream, so that a benchmark can state how many
 * of the library's kernels one call launches.  Returns the count, or a
 * negative status (SA_ERR_NULL for a NULL graph, SA_ERR_LAUNCH if the graph
 * cannot be read).
 */
int sa_graph_kernel_count(void* graph);

/*
 * sa_check_wait_timeout -- diagnostic (no counterpart on the pages): runs the
 * library's bounded-wait timeout path on purpose, without a fault.
 *
 * Every pipelined kernel waits on its shared-memory barriers for at most about
 * 2e9 SM cycles (about one second), then ORs SA_ERRBIT_TIMEOUT into the
 * caller's error word, sets its CTA's abort flag and returns, leaving the
 * context usable.  A correct call never takes that path; this call makes one
 * warp wait on a barrier that nothing arrives on (no copy or MMA in flight),
 * then wait once more on the abort flag the first wait set.
 *
 * err_word: device pointer to one uint32 (zeroed by the caller), receives
 *           SA_ERRBIT_TIMEOUT.
 * out:      device pointer to four uint32: [0] 1 if the first wait gave up,
 *           [1] 1 if the second returned at once, [2], [3] the first wait's
 *           SM cycles (low, high word).
 * stream:   cudaStream_t or NULL.  Asynchronous; about one second of device
 *           time on one SM.
 * Returns SA_OK, SA_ERR_NULL, SA_ERR_ALIGN (a pointer not 4-byte aligned) or
 * SA_ERR_LAUNCH.
 */
int sa_check_wait_timeout(uint32_t* err_word, uint32_t* out, void* stream);

/*
 * validate_indices -- [IS] validate_indices / validate_index_rows.
 *
 * idx: [B, I, Sq, K] int32 (idx_is_i64 = 0) or int64 (idx_is_i64 = 1).
 * Each row is scanned left to right: -1 marks padding; any other value is
 * checked, in this order, for being below -1, following padding, being
 * >= bound, equal to its predecessor, smaller than it.  The first failing
 * column decides the row's code; a row of only -1 is SA_IDX_ALL_PADDING.
 * bound_per_batch: nullable device int64 [B]; when NULL every row is bounded
 * by `bound`.
 * row_status: nullable device uint8 [B*I*Sq], written with each row's code
 * (0 = valid).  err_word: device uint32, OR-ed with every row's code (the
 * caller zeroes it).  Bit-exact with the definition.
 */
int validate_indices(const void* idx, int idx_is_i64, int64_t B, int64_t I, int64_t Sq,
                     int64_t K, const int64_t* bound_per_batch, int64_t bound,
                     uint8_t* row_status, uint32_t* err_word, void* stream);

/*
 * build_present_kv -- [IS] build_present, [SA] build_kv.  A pure copy
 * (bit-exact), for K and (optionally) V in one launch.
 *
 * Concat mode (write_pos == NULL):
 *   present[b,h,t,:] = past[b,h,t,:]      for t <  P   (past is [B,H,P,D])
 *                    = cur[b,h,t-P,:]     for P <= t < P+C (cur is [B,H,C,D])
 *   present is [B, H, present_stride, D] with present_stride >= P + C;
 *   positions >= P + C are not written.  past may be NULL only when P == 0.
 *   present must not overlap past or cur (SA_ERR_OVERLAP).
 * Append mode (write_pos != NULL, device int64 [B]):
 *   present is a capacity cache [B, H, present_stride, D]; cur[b,h,c,:] is
 *   written at position write_pos[b] + c.  past must be NULL or equal to
 *   present (in place: nothing else moves); another past [B,H,present_stride,D]
 *   is first copied whole.  A write_pos outside [0, present_stride - C] skips
 *   that batch and sets SA_ERRBIT_WRITE_POS in err_word (nullable).
 * past_v/cur_v/present_v: the same for V; present_v NULL means K only.
 * dtype: SA_F32, SA_F16 or SA_BF16 (any 2/4-byte element copies exactly).
 */
int build_present_kv(const void* past_k, const void* cur_k, void* present_k,
                     const void* past_v, const void* cur_v, void* present_v, int dtype,
                     int64_t B, int64_t H, int64_t P, int64_t C, int64_t D,
                     int64_t present_stride, const int64_t* write_pos, uint32_t* err_word,
                     void* stream);

/*
 * Selected-token attention -- [IS] index_share_row (semantics), [SA]
 * Semantics + attention_split/attention_combine (split-KV, fixed-order
 * combine), [CSA] dense window + FP8 records + sink.
 *
 * For every output row (b, h, i) with kvh = h / (Hq/Hkv) and index head
 * ih = 0 (I == 1), kvh (I == Hkv) or h (I == Hq):
 *   C = valid prefix of idx[b, ih, i, :] (entries before the first -1);
 *   with window W > 0: C = [len_b - W, len_b) united with {j in C : j < len_b - W};
 *   s_j = scale * q . k_j;  s_j = softcap * tanh(s_j / softcap) if softcap != 0;
 *   s_j += bias(b, h, i, j) when bias != NULL ([IS] index_share_row / bias_at:
 *         keyed by the cache position j);
 *   s_j = -inf when j >= len_b (len_b = kv_len[b], or T), or causal and
 *         j > past_len + i;
 *   y = sum_j softmax(s)_j v_j, with exp(sink[h] - max) added to the
 *   denominator when sink != NULL; a row whose scores are all -inf gives 0.
 * Layouts:
 *   q  [B, Hq, Sq, D] in q_dtype (F32, F16, BF16);  y [B, Hq, Sq, Dv] same dtype.
 *   dense cache (kv_dtype == q_dtype): k_cache [B, Hkv, T, D], v_cache [B, Hkv, T, Dv].
 *   FP8 cache (kv_dtype SA_FP8_E4M3_B64, q_dtype BF16): k_cache is
 *     [B, Hkv, T, record_stride] bytes, each record (D - n_rope)/64 blocks of
 *     [E8M0 scale, 64 E4M3FN codes] then n_rope little-endian bf16 values;
 *     V is the same decoded record (its first Dv dims); v_cache is ignored.
 *   idx [B, I, Sq, K] int32 or int64.  kv_len: nullable device int64 [B].
 *   sink: nullable device float [Hq] (natural-log logits).
 *   bias: nullable device float32, dense row-major of shape
 *     bias_dims[0 .. bias_rank-1] with 0 <= bias_rank <= 4, broadcast against
 *     [B, Hq, Sq, T] from the right ([IS] validate_bias_shape: every axis is 1
 *     or the extent it lines up with; otherwise SA_ERR_SHAPE).  Entries are
 *     finite or -inf (a -inf masks its key); the bias counts only for the
 *     candidate keys, each read at its cache position.
 * options: 0, or SA_OPT_* bits choosing a kernel variant (the result is the
 * same operation; tests use them to cover every path).
 * scale: 0 means 1/sqrt(D).  Index rows are validated on the device against
 * len_b when err_word != NULL (row_status nullable, as in validate_indices);
 * malformed rows never fault: negative entries are skipped, entries >= len_b
 * are masked, and the other entries of such a row (after padding, repeated or
 * out of order) are attended as they stand.  A malformed row's output is
 * finite; only a well-formed row's output is the definition above.
 * Fused append (dense cache only): when k_cur != NULL, the current token(s)
 * k_cur / v_cur [B, Hkv, cur_len, D] are first written into the cache at
 * positions write_pos[b] .. write_pos[b] + cur_len - 1 (write_pos: nullable
 * device int64 [B], NULL meaning T - cur_len) -- build_present_kv's append
 * mode -- and attention sees them there.  A write position outside
 * [0, T - cur_len] sets SA_ERRBIT_WRITE_POS and skips that batch's write.
 * Workspace: sparse_attn_decode_workspace(p) bytes, 256-byte aligned; its
 * contents on entry do not matter (every word is written before it is read).
 * It holds the planned candidate positions and the key splits' partial
 * results; for the FP8 cache with Hq a multiple of 128 also the decoded
 * candidates (B * Sq * ceil((window + K) / 128) * 128 rows of D bf16 values,
 * e.g. 40 MB for B 16, 2176 candidates, D 576).  Calls that share a workspace
 * must not overlap on the GPU.
 */
typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* idx;
  const float* sink;
  void* y;
  int32_t q_dtype;
  int32_t kv_dtype;
  int32_t idx_is_i64;
  int32_t causal;
  int64_t B, Hq, Hkv, Sq, D, Dv, T, I, K;
  const int64_t* kv_len;
  int64_t past_len;
  float scale;
  float softcap;
  int64_t window;
  int64_t record_stride;
  int64_t n_rope;
  uint32_t* err_word;
  uint8_t* row_status;
  const void* k_cur;
  const void* v_cur;
  const int64_t* write_pos;
  int64_t cur_len;
  void* workspace;
  size_t workspace_bytes;
  const float* bias;
  int64_t bias_rank;
  int64_t bias_dims[4];
  uint32_t options;
  uint32_t reserved_;   /* must be 0 */
} sa_sparse_params;

size_t sparse_attn_decode_workspace(const sa_sparse_params* p);
int sparse_attn_decode(const sa_sparse_params* p, void* stream);

/*
 * sparse_attn_decode_noalloc -- the same operation as sparse_attn_decode for
 * callers that cannot allocate device memory themselves: runtimes that own a
 * fixed device-memory budget and account for every byte, plugins whose host
 * framework passes them inputs and outputs but no scratch, or code that must
 * not set off cudaMalloc's implicit device synchronisation (or be refused it
 * during a global-mode stream capture).  The pages have no counterpart: it is
 * a deployment variant of this library's own entry point.
 *
 * p->workspace / p->workspace_bytes are ignored.  Scratch comes from one
 * built-in device buffer of SA_NOALLOC_SCRATCH_BYTES, which every GPU that
 * loads the library holds until the process exits; a request needing more
 * (sparse_attn_decode_workspace(p) > SA_NOALLOC_SCRATCH_BYTES) returns
 * SA_ERR_SCRATCH_LIMIT before anything is enqueued.  Nothing is allocated or
 * freed.  The first call on each device looks up that buffer's device
 * address (once, with that device current); make that first call before any
 * stream capture.  The address is kept for the life of the process: a device
 * reset (cudaDeviceReset) while the library is loaded is not supported by this
 * entry point, since the kept address would then be stale.  Every call
 * shares the buffer and it keeps the last call's contents (the call needs
 * none of it cleared: all scratch is written before it is read), so calls
 * that overlap on the GPU -- on different streams, or from different
 * threads, of the same device -- race and must be serialised by the caller.
 */
#define SA_NOALLOC_SCRATCH_BYTES (16u << 20)
int sparse_attn_decode_noalloc(const sa_sparse_params* p, void* stream);

/*
 * sparse_index_select -- ratio-4 index scoring and top-k selection, the step
 * that produces the selected indices: [CSA-CPU] finalize_index_query,
 * hadamard_bf16, fp4_roundtrip, select_ratio4_topk; [CSA]
 * csa_ratio4_index_select, csa_ratio4_index_replicate.
 *
 * For each row (b, s), at position p = query_start (or query_start_b[b]) + s:
 *   q_h = fp4_roundtrip(hadamard_bf16(bf16(query[b, s, h, :])))   per head h,
 *     the Walsh-Hadamard transform with a 1/sqrt(ID) scale rounded to bf16,
 *     then every block of 32 rounded to FP4 E2M1 with an E8M0 scale by the
 *     OCP MX rule (scale 2^(floor(log2 amax) - 2), nearest value, ties to
 *     even, saturating);
 *   score_r = sum_h relu(q_h . k_r) * weight[b, s, h] * c,  c = (1/sqrt(ID))/sqrt(IH),
 *     for the causal records r < min(R, (p + 1) / 4), in binary32: each dot
 *     product summed in ascending dimension order, the heads in ascending
 *     order, every multiply and add rounded on its own (the pages' order; the
 *     result is that definition bit for bit);
 *   the records ranked by score (Rust f32::total_cmp, higher first) and then
 *   by record index; the first topk written, -1 after them.
 * The compressed RoPE of the query's last components is the caller's: the
 * query enters after it.
 *
 * query: float32 [B, S, IH, ID], ID in {32, 64, 128, 256}; weight: float32
 * [B, S, IH]; keys: [B, R, key_stride] bytes, each record ID/32 blocks of
 * [E8M0 scale byte, 16 bytes of E2M1 codes, element 2j in the low nibble of
 * byte j] (68 bytes for ID 128), key_stride a multiple of 4, keys 4-byte
 * aligned.  selected: int32 [B, out_heads, S, topk], the same row for every
 * output head ([CSA] replicate); ascending = 1 writes the selected records
 * in ascending record order instead of score order (the form
 * sparse_attn_decode validates).  1 <= topk <= 4096, 1 <= IH <= 256.
 * row_status (nullable uint8 [B*S]) and err_word (nullable): SA_SEL_TIE when
 * two scores of the row are equal (the pages refuse such input; the ranking
 * still orders them by record), SA_SEL_NONFINITE when a score is NaN or
 * infinite; err_word receives them shifted into SA_ERRBIT_SEL_*.
 * Workspace: sparse_index_select_workspace(p) bytes, 256-byte aligned,
 * contents on entry irrelevant.  Deterministic.
 */
#define SA_SEL_TIE 1
#define SA_SEL_NONFINITE 2
#define SA_ERRBIT_SEL_TIE 512
#define SA_ERRBIT_SEL_NONFINITE 1024
typedef struct {
  const float* query;
  const float* weight;
  const uint8_t* keys;
  int32_t* selected;
  uint8_t* row_status;
  uint32_t* err_word;
  int64_t B, S, IH, ID, R, topk, key_stride, out_heads;
  int64_t query_start;
  const int64_t* query_start_b;
  int32_t ascending;
  int32_t reserved_;    /* must be 0 */
  void* workspace;
  size_t workspace_bytes;
} sa_index_select_params;

size_t sparse_index_select_workspace(const sa_index_select_params* p);
int sparse_index_select(const sa_index_select_params* p, void* stream);

/*
 * csa_ratio4_attention -- compressed sparse attention, ratio 4, in the pages'
 * own form: [CSA-CPU] ratio4_attention (with its call in execute_ratio4),
 * [CSA] csa_ratio4_sink_attention.
 *
 * For query s of batch b at position p = total - S + s, with base = total - L
 * (the position of current_kv row 0):
 *   dense slots c < dense (dense = 128, or min(L, 128) when total == S): the
 *     current_kv row at position max(base, p + 1 - 128) + c when that is <= p
 *     and stored (row < L), else no candidate;
 *   slot dense + k: selected record selected[b, s, k] when it lies in
 *     [0, min(R, total / 4)); a negative entry is no candidate, one at or past
 *     that bound is skipped and sets SA_ERRBIT_RECORD (err_word nullable);
 *   score = scale * q . row + bias(b, h, s, slot) (bias nullable, float32,
 *     rank <= 4, broadcast right-aligned against [B, H, S, dense + topk]);
 *   y = sum softmax(score) row, with exp(sink[h] - max) added to the
 *     denominator (sink nullable); a query with no candidate gives 0.
 * K = V = the row: current_kv is one latent head; a record decodes as
 * (D - n_rope) / 64 blocks of [E8M0 scale, 64 E4M3FN] then n_rope LE bf16
 * (583 bytes at D 512, n_rope 64; any byte alignment).
 * Layouts: query / y [B, S, H, D] (q_dtype SA_F32 or SA_BF16, y the same);
 * current_kv [B, L, D] (kv_dtype SA_F32 or SA_BF16); records [B, R,
 * record_stride] bytes; selected int32 [B, S, topk].  D 128 or 512, H a
 * multiple of 32, n_rope even with D - n_rope a positive multiple of 64.
 * Arithmetic: rows and queries as bf16 (float inputs rounded; FP8 records
 * exact) on the tensor cores with fp32 accumulation and softmax.
 * Workspace: csa_ratio4_attention_workspace(p) bytes, 256-byte aligned,
 * contents on entry irrelevant (the candidate rows, B * S * (dense + topk)
 * rows of D bf16, and split partials).
 */
typedef struct {
  const void* query;
  const void* current_kv;
  const uint8_t* records;
  const int32_t* selected;
  const float* sink;
  const float* bias;
  int64_t bias_rank;
  int64_t bias_dims[4];
  void* y;
  int32_t q_dtype;
  int32_t kv_dtype;
  int64_t B, S, H, D, n_rope, L, R, topk, record_stride, total;
  float scale;          /* 0: 1/sqrt(D) */
  int32_t reserved_;    /* must be 0 */
  uint32_t* err_word;
  void* workspace;
  size_t workspace_bytes;
} sa_csa_params;

size_t csa_ratio4_attention_workspace(const sa_csa_params* p);
int csa_ratio4_attention(const sa_csa_params* p, void* stream);

/*
 * csa_ratio128_compress / csa_ratio4_main_compress / csa_ratio4_index_compress
 * -- the compression stages that produce the CSA records: [CSA-CPU]
 * compress_ratio4_stream, pool_ratio4_record, pool_ratio128_record,
 * finalize_attention_record, finalize_index_record, apply_compressed_rope;
 * [CSA] csa_ratio128_compress, csa_ratio4_main_compress,
 * csa_ratio4_index_compress.
 *
 * One call appends S tokens per sequence at positions start = total - S ..
 * total - 1.  Token p's score row is gate + ape[p % ratio].  Every block of
 * `ratio` tokens that closes in [start, total) emits record k = p / ratio
 * (p its last token), computed at block_start = k * ratio:
 *   pool: per dimension d, over the candidates in order -- ratio 128: the
 *     block's 128 tokens; ratio 4: the previous block's 4 tokens on source
 *     dim d, then the block's 4 tokens on source dim D + d (a token before
 *     position 0 is no candidate) -- the weighted mean sum(w v) / sum(w)
 *     with w = e^(score - max score) (the binary32 rounding of the exact
 *     value), candidates of score -inf left out; then bf16;
 *   RMSNorm: binary32 square sum in dimension order, times
 *     1 / sqrt(sum / D + 1e-6), times norm[d], bf16;
 *   compressed RoPE of the last n_rope dims, pair i = dims (D - n_rope + 2i,
 *     +1): frequency f = b (1 - r) + (b / 16) r with b = 160000^(-2i/n_rope)
 *     and r = clamp((i - 15) / 10, 0, 1), angle = block_start * f (binary32),
 *     cos and sin rounded from their exact values; each component bf16;
 *   attention records (main, ratio 128): (D - n_rope) / 64 blocks of
 *     [E8M0 byte, 64 E4M3FN codes] -- the block exponent is the smallest e
 *     with amax / 2^e <= 448 (0 for a zero block), codes the nearest-even
 *     E4M3FN of x / 2^e -- then the n_rope dims as little-endian bf16:
 *     (D - n_rope) / 64 * 65 + 2 n_rope bytes (583 at D 512, n_rope 64);
 *   index keys: the Walsh-Hadamard transform (butterflies of span 1, 2, 4,
 *     ..., then times 1 / sqrt(D), bf16), then D / 32 blocks of [E8M0 byte,
 *     16 bytes of FP4 E2M1 codes, even element in the low nibble] with the
 *     OCP MX scale 2^(floor(log2 amax) - 2) (byte 0 for a zero block):
 *     D / 32 * 17 bytes (68 at D 128).
 * Every step is one binary32 operation rounded to nearest, in this order.
 * A record that meets a non-finite value (no finite score in a dimension,
 * an unusable sum, a non-finite square sum or result) is stored as zeros and
 * sets SA_ERRBIT_COMPRESS in err_word (nullable).
 *
 * Layouts (float32 unless stated): kv, gate [B, S, W] with W = D (ratio
 * 128) or 2 D (ratio 4); ape [ratio, W]; norm [D]; carry [B, slots, 2, W]
 * with slots 128 (ratio 128) or 8 (ratio 4), channel 0 the value and 1 the
 * score, read and rewritten in place: it holds the open block's tokens (slot
 * p % 128, or 4 + p % 4) and, at ratio 4, the last closed block's (slots
 * 0..3); empty slots hold (0, -inf).  A call with start == 0 ignores the
 * carry's contents.  records [B, rows, record_stride] bytes and logical
 * [B, rows, D] (the record's dequantized values), each nullable but not
 * both: row k is written, the others untouched.  rows >= total / ratio.
 * Shapes: attention records need D % 4 == 0, D <= 1024, (D - n_rope) % 64
 * == 0; index keys D in {32, 64, 128, 256}; n_rope even, <= min(D, 128).
 * kv, gate, ape and carry 16-byte aligned.  No workspace.
 */
typedef struct {
  const float* kv;
  const float* gate;
  const float* ape;
  const float* norm;
  float* carry;
  uint8_t* records;
  float* logical;
  uint32_t* err_word;
  int64_t B, S, D, n_rope, rows, record_stride, total;
  int64_t reserved_;  /* must be 0 */
} sa_compress_params;

int csa_ratio128_compress(const sa_compress_params* p, void* stream);
int csa_ratio4_main_compress(const sa_compress_params* p, void* stream);
int csa_ratio4_index_compress(const sa_compress_params* p, void* stream);

/*
 * csa_pool_weight -- w[i] = e^t[i] rounded to binary32 (nearest even), the
 * pool weight of the compression stages, for checking that rounding on its
 * own: t, w device float32 [n] (t <= 0 is the compression's domain; any
 * value is accepted).  Returns SA_OK or an argument error.
 */
int csa_pool_weight(const float* t, float* w, int64_t n, void* stream);

/* attention-mask element types of sa_prefill_params.mask_kind */
#define SA_MASK_NONE 0
#define SA_MASK_F32 1
#define SA_MASK_F16 2
#define SA_MASK_BF16 3
#define SA_MASK_BOOL 4  /* one byte per element: nonzero keeps the key */

/*
 * attn_prefill -- [SA] Semantics with no past: q [B, Hq, S, D],
 * k/v [B, Hkv, S, D] (GQA, Hq % Hkv == 0), y [B, Hq, S, D]; query i sees
 * keys 0..i when causal; softcap as above, applied before the mask; fp32
 * softmax.  present_k / present_v (nullable, [B, Hkv, S, D]) receive exact
 * copies of k / v (past ++ current with an empty past).  dtype: SA_BF16 or
 * SA_F16, or SA_F32.  Workspace rules as for sparse_attn_decode.
 * bf16 / f16 with D in {64, 128}, a positive scale and 16-byte aligned
 * q / k / v / y run on the tcgen05 tensor-core kernel and need no workspace
 * (a misaligned y there is SA_ERR_ALIGN); other shapes take the general
 * kernel.  err_word (nullable) receives SA_ERRBIT_TIMEOUT if the tensor-core
 * pipeline stalled, in which case y is unspecified.
 * nonpad_kv_seqlen (nullable device int64 [B]; [SA] attention_row's padding
 * frontier): keys j >= nonpad[b] are masked (a negative entry disables that),
 * and a causal query i then sees keys j <= i + nonpad[b] - S; a row left with
 * no key gives 0.  Served by the tcgen05 kernel.
 * attn_mask (nullable device, [SA] mask_bias): mask_kind elements in a dense
 * row-major tensor of shape mask_dims[0 .. mask_rank-1], rank <= 4, broadcast
 * right-aligned against [B, Hq, S, S] (every axis but the last 1 or its
 * target; the last is the key axis: keys at or past its extent take -inf);
 * float masks add their value after the softcap, bool masks keep a key where
 * nonzero.  A request with a mask runs on the per-row kernels (correct, not
 * tuned) and writes present K/V by a separate copy.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  void* y;
  void* present_k;
  void* present_v;
  int32_t dtype;
  int32_t causal;
  int64_t B, Hq, Hkv, S, D;
  float scale;
  float softcap;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* err_word;   /* nullable: SA_ERRBIT_TIMEOUT if a tensor-core pipeline stalled */
  const void* attn_mask;
  int32_t mask_kind;    /* SA_MASK_NONE / _F32 / _F16 / _BF16 / _BOOL */
  int32_t reserved_;    /* must be 0 */
  int64_t mask_rank;
  int64_t mask_dims[4];
  const int64_t* nonpad_kv_seqlen;
} sa_prefill_params;

size_t attn_prefill_workspace(const sa_prefill_params* p);
int attn_prefill(const sa_prefill_params* p, void* stream);

/*
 * paged_attn_decode -- [PG] paged causal decode.  One new query per
 * sequence: q [B, Hq, D], y [B, Hq, D].  Pools k_pool / v_pool are
 * [num_pages, Hkv, page_tokens, D]; token t of sequence b lives at page
 * block_table[b * max_pages + t / page_tokens], slot t % page_tokens.
 * ctx_len[b] (device int32) counts the new token, which attends to all
 * ctx_len[b] tokens.  If k_new / v_new ([B, Hkv, D]) are given they are first
 * written into the pool at token ctx_len[b] - 1.  A ctx_len outside
 * [1, max_pages*page_tokens] or a table entry outside [0, num_pages) sets
 * SA_ERRBIT_PAGE (err_word nullable) and is never dereferenced.
 * dtype SA_F16 / SA_BF16 / SA_F32; scale 0 means 1/sqrt(D).  Workspace rules
 * as for sparse_attn_decode.
 */
typedef struct {
  const void* q;
  void* k_pool;
  void* v_pool;
  const void* k_new;
  const void* v_new;
  const int32_t* block_table;
  const int32_t* ctx_len;
  void* y;
  int32_t dtype;
  uint32_t options;     /* 0, or SA_OPT_ROW_COPIES (pages fetched row by row) */
  int64_t B, Hq, Hkv, D, page_tokens, max_pages, num_pages;
  float scale;
  float pad2_;
  uint32_t* err_word;
  void* workspace;
  size_t workspace_bytes;
} sa_paged_params;

size_t paged_attn_decode_workspace(const sa_paged_params* p);
int paged_attn_decode(const sa_paged_params* p, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_H */
