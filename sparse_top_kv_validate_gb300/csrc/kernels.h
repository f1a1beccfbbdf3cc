// kernels.h -- argument blocks and launchers shared between the host entry
// points (sa_api.cu) and the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

// ---- index validation --------------------------------------------------------
struct ValidateArgs {
  const void* idx;
  int is_i64;
  int vec_ok;                 // 16-byte vector loads are legal
  int64_t rows;               // B * I * Sq
  int64_t rows_per_batch;     // I * Sq
  int64_t K;
  const int64_t* bound_per_batch;
  int64_t bound;
  uint8_t* row_status;
  uint32_t* err_word;
};
int launch_validate(const ValidateArgs& a, cudaStream_t st);

// ---- present KV --------------------------------------------------------------
struct PresentArgs {
  const void* past[2];
  const void* cur[2];
  void* present[2];
  int n_tensors;              // 1 (K) or 2 (K and V)
  int esz;                    // element bytes
  int64_t B, H, P, C, D;
  int64_t stride;             // present positions per (b, h)
  const int64_t* write_pos;   // append mode when non-null
  int copy_past;              // append mode: copy past wholly first
  uint32_t* err_word;
};
int launch_present(const PresentArgs& a, cudaStream_t st);

// ---- per index row plan: validation + candidate positions + append ----------------
struct PlanArgs {
  const void* idx;            // [B, I, Sq, K]
  int idx_is_i64;
  int vec_ok;                 // 16-byte vector loads are legal
  int plan_rows;              // 0: append blocks only
  int write_positions;        // write pos (0: the consumer plans its own positions)
  int validate;               // write row_status / err_word
  int causal;
  int64_t B, I, Sq, K, T, window, past_len;
  int64_t n_cand_pad;         // positions per row: (window + K) rounded up to 16
  const int64_t* kv_len;      // nullable
  int32_t* pos;               // [B*I*Sq, n_cand_pad] cache positions or -1
  uint8_t* row_status;
  uint32_t* err_word;
  // fused append of the current token(s) (append_blocks == 0: none)
  const void* k_cur;
  const void* v_cur;
  void* k_cache;
  void* v_cache;
  const int64_t* write_pos;   // nullable: T - C
  int64_t Hkv, C, D;
  int esz;
  int append_blocks;
};
int launch_plan(const PlanArgs& a, cudaStream_t st);

// ---- gather decode (sparse and paged) ------------------------------------------
enum KeySource : int { kSparse = 0, kPaged = 1, kDense = 2 };
enum BiasKind : int { kBiasF32 = 0, kBiasF16 = 1, kBiasBF16 = 2, kBiasBool = 3 };

struct GatherArgs {
  // tensors
  const void* q;              // [B, Hq, Sq, D]
  const void* k;              // dense cache or page pool
  const void* v;
  void* y;                    // [B, Hq, Sq, Dv]
  const float* sink;          // nullable [Hq]
  const void* bias;           // nullable: additive bias / attention mask, element
  int64_t bias_sb, bias_sh;   //   (b,h,i,j) at b*bias_sb + h*bias_sh + i*bias_si +
  int64_t bias_si, bias_sk;   //   j*bias_sk (broadcast axes have stride 0)
  int bias_kind;              // kBiasF32 / kBiasF16 / kBiasBF16 / kBiasBool
  int64_t bias_key_extent;    // > 0: keys j >= it take -inf (a short mask key axis)
  const int64_t* dense_nonpad;  // dense source: nullable per-batch padding frontier
  float* part_o;              // unnormalised partial outputs (layout per kernel)
  float* part_ml;             // partial running max (log2 units) and sum
  uint32_t* err_word;
  // geometry
  int source;                 // KeySource
  int64_t B, Hq, Hkv, Sq, D, Dv;
  int64_t g;                  // Hq / Hkv
  int64_t hpu;                // heads served per unit
  int64_t n_groups;           // units per (b, i): Hkv, or Hq when rows are per head
  int64_t units;              // B * n_groups * Sq
  int64_t splits;             // SIMT path: key splits per unit
  int64_t chunk;              // SIMT path: candidates per split
  int64_t n_cand;             // candidates per unit (upper bound for paged)
  int64_t tiles_per_unit;     // stream kernel, sparse/dense: ceil(n_cand / 16)
  int64_t tiles_per_warp;     // stream kernel, sparse/dense: tiles per warp range
  const int32_t* pos;         // stream kernel, sparse: planned cache positions
  int64_t n_cand_pad;         // positions per planned row
  int64_t* meta;              // stream kernel -> combine: [0] tiles per warp
  int32_t* pref_out;          // stream kernel -> combine (paged): tile prefix [B+1]
  // sparse source
  const void* idx;
  int idx_is_i64;
  int64_t I, K, T;            // index heads, index width, cache stride
  int64_t window;
  const int64_t* kv_len;      // nullable
  int64_t past_len;
  int causal;
  // fused current-token append (sparse source; k_cur nullable)
  const void* k_cur;          // [B, Hkv, C, D]
  const void* v_cur;
  const int64_t* write_pos;   // nullable: T - C
  int64_t C;
  // paged source
  const int32_t* block_table;
  const int32_t* ctx_len;
  int64_t page_tokens, max_pages, num_pages;
  // FP8 hybrid records (sparse source)
  int64_t record_stride;      // bytes between records
  void* fp8_kdec;             // tcgen05 FP8 path: decoded rows [units, n_cand_pad, 576] bf16
  int fp8_own_positions;      // tcgen05 FP8 path: the decode kernel writes pos itself
  int fp8_after_plan;         //   and the plan kernel (validation only) runs just before it
  int row_copies;             // stream kernel: per-row bulk copies, no tensor maps
  int fp8_warp_mma;           // FP8 records: the warp-level MMA kernel only
  void* ev_before;            // nullable cudaEvent_t pair recorded around the dominant kernel
  void* ev_after;
  // math
  float scale_log2;           // scale * log2(e)
  float softcap;              // 0 = off
  float inv_softcap;
};

// SIMT split-K kernel (any dtype, D <= 512) + its combine kernel.
int launch_gather_simt(const GatherArgs& a, int dtype, cudaStream_t st);
int launch_combine(const GatherArgs& a, int dtype, cudaStream_t st);
// Whether the persistent tensor-core stream kernel serves this request.
bool gather_uses_mma(const GatherArgs& a, int dtype);
// Persistent tensor-core stream kernel (f16/bf16, D in {64,128,256}).
size_t stream_smem_bytes(int D, int source, int64_t B);
int stream_warps(int D);
int stream_max_batch_paged();
int launch_gather_stream(const GatherArgs& a, int dtype, int grid, cudaStream_t st);
// FP8 hybrid-record decode (MQA, D = 512 E4M3 + 64 bf16, bf16 Q/Y).
size_t fp8_smem_bytes();
int fp8_chunk_tiles_max();
int launch_fp8_decode(const GatherArgs& a, cudaStream_t st);
// The same on the fifth-generation tensor cores for blocks of 128 query heads:
// a gather kernel decodes the planned candidates' records into fp8_kdec, then
// the attention kernel streams them by TMA (planned positions padded to
// 128-key tiles, at most fp8_tc_max_tiles() tiles per key split).
bool fp8_tc_supported(const GatherArgs& a);
int fp8_tc_max_tiles();

// One warp waits on a barrier that nothing arrives on (k_diag.cu).
int launch_wait_timeout(uint32_t* err_word, uint32_t* out, cudaStream_t st);
size_t fp8_tc_decoded_row_bytes();
// Key splits that the attention kernel merges itself (a cluster of `splits`
// CTAs per output block, `blocks` such clusters resident at once); otherwise
// partials for launch_combine.
bool fp8_tc_cluster_merge(int64_t splits, int64_t blocks);
int launch_fp8_tc(const GatherArgs& a, cudaStream_t st);
// Merge of the units the stream kernel split across warps.
int launch_stream_combine(const GatherArgs& a, int dtype, cudaStream_t st);

// ---- dense prefill on the fifth-generation tensor cores (tcgen05 + TMEM + TMA) ------
// Records ev (a cudaEvent_t, nullable) on st: the measurement hook.
inline void mark_event(void* ev, cudaStream_t st) {
  if (!ev) return;
  // under stream capture only an external record becomes a node of the graph
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), st);
}

struct PrefillTcArgs {
  const void* q;              // [B, Hq, S, D]
  const void* k;              // [B, Hkv, S, D]
  const void* v;
  void* y;                    // [B, Hq, S, D]
  void* present_k;            // nullable: [B, Hkv, S, D] copy of k, written by the kernel
  void* present_v;            // nullable: copy of v
  int dtype;                  // SA_BF16 or SA_F16
  int causal;
  int64_t B, Hq, Hkv, S, D;
  float scale;                // > 0
  float softcap;              // 0 = off
  uint32_t* err_word;         // nullable: SA_ERRBIT_TIMEOUT on a stalled pipeline
  const int64_t* nonpad;      // nullable [B]: keys >= nonpad[b] masked, causal offset nonpad[b] - S
};
bool prefill_tc_supported(const PrefillTcArgs& a);
int launch_prefill_tc(const PrefillTcArgs& a, cudaStream_t st);

// ---- ratio-4 index scoring and top-k selection ----------------------------------------
constexpr int kQinfoZero = 1;             // index-query head whose codes are all zero
constexpr int kQinfoNonfinite = 2;        // index-query head with a non-finite block
constexpr int kSelTie = 1;                // row status: equal scores in the row
constexpr int kSelNonfinite = 2;          // row status: a score is NaN or infinite
constexpr int kSelErrShift = 9;           // row status << shift = err_word bits

struct IndexArgs {
  const float* query;         // [rows, IH, ID], rows = B * S
  const float* weight;        // [rows, IH]
  const uint8_t* keys;        // [B, R, key_stride]
  int32_t* selected;          // [B, out_heads, S, topk]
  uint8_t* row_status;        // nullable [rows]
  uint32_t* err_word;         // nullable
  int64_t rows, S, IH, ID, R, topk, key_stride, out_heads;
  int64_t query_start;
  const int64_t* query_start_b;  // nullable [B]
  int ascending;              // 1: records in ascending order, else score order
  float had_scale;            // 1 / sqrt(ID) in binary32
  float weight_scale;         // (1 / sqrt(ID)) / sqrt(IH) in binary32
  // workspace
  int8_t* qcodes;             // [rows, IH, ID] signed 2 * E2M1 codes
  int8_t* qexp;               // [rows, IH, ID / 32] block exponents (127: non-finite)
  int4* qinfo;                // [rows, IH] {exponent range, min, max, zero / non-finite}
  float* qscale;              // [rows, IH, ID / 32] 2^(block exponent)
  float* scores;              // [rows, R]
  uint32_t* hist;             // [rows, 2048] counts of the rank keys' top 11 bits
  uint32_t* rowflags;         // [rows] SEL_TIE / SEL_NONFINITE found while scoring
  uint32_t* done;             // [rows] CTAs of the selection kernel finished with the row
  unsigned long long* bucket; // [rows, R] (rank key, record) of the threshold bin
  int hash_slots;             // equal-score hash set: power of two >= 2 R, in parts
  int hash_log2;
  int sel_slots;              // next power of two >= topk
  void* ev_before;            // nullable measurement events around the score kernel
  void* ev_after;
};
size_t index_topk_smem_bytes(int64_t sel_slots);
size_t index_tie_smem_bytes(int hash_slots);
size_t index_score_smem_bytes(int64_t IH, int64_t ID, int64_t key_stride);
int launch_index_select(const IndexArgs& a, cudaStream_t st);

// ---- compressed sparse attention (ratio 4), the pages' own form ------------------------
struct CsaArgs {
  const void* query;          // [B, S, H, D] (q_dtype)
  const void* window;         // current_kv [B, L, D] (kv_dtype)
  const uint8_t* records;     // [B, R, record_stride] hybrid FP8
  const int32_t* selected;    // [B, S, topk]
  const float* sink;          // nullable [H]
  const float* bias;          // nullable: element (b,h,s,slot) at b*sb + h*sh + s*si + slot*sk
  int64_t bias_sb, bias_sh, bias_si, bias_sk;
  void* y;                    // [B, S, H, D] (q_dtype)
  int q_dtype, kv_dtype;
  int64_t B, S, H, D, n_rope, L, R, topk, record_stride, total;
  int64_t dense;              // dense slots: 128, or min(L, 128) when the block starts at 0
  int64_t valid_records;      // min(R, total / 4)
  int64_t c_pad;              // candidate slots, rounded up to 16 (128 on the tensor-core path)
  int64_t splits, chunk_tiles;  // chunk_tiles: 16-slot tiles, or 128-slot tiles when tc
  int tc;                     // the tcgen05 attention kernel (k_fp8_tc.cu) instead of csa_attn_kernel
  float scale_log2;
  uint32_t* err_word;
  // workspace
  __nv_bfloat16* rows;        // [B * S, c_pad, D] candidate rows
  uint8_t* valid;             // [B * S, c_pad]
  float* part_o;              // [B * S, splits, H, D] when splits > 1
  float* part_ml;             // [B * S, splits, H, 2]
  void* ev_before;            // nullable measurement events around the attention kernel
  void* ev_after;
};
size_t csa_attn_smem_bytes(int64_t D);
int launch_csa(const CsaArgs& a, cudaStream_t st);
// tcgen05 attention over the assembled rows (D = 512, 128-head blocks, bf16 queries)
bool csa_tc_supported(int64_t D, int64_t H, int q_dtype);
int csa_tc_max_tiles();
// *merged: the key splits were merged on chip (no combine kernel needed)
int launch_csa_tc(const CsaArgs& a, cudaStream_t st, bool* merged);

// ---- CSA compression stages (ratio 4 records / index keys, ratio 128) -------------------
constexpr int kCompressAttn = 0;   // hybrid FP8 attention record
constexpr int kCompressIndex = 1;  // FP4 index key

struct CompressArgs {
  const float* kv;            // [B, S, W] source values (W = D at ratio 128, 2 D at ratio 4)
  const float* gate;          // [B, S, W] source scores
  const float* ape;           // [ratio, W]
  const float* norm;          // [D]
  float* carry;               // [B, slots, 2, W], slots 128 or 8
  uint8_t* records;           // nullable [B, rows, record_stride]
  float* logical;             // nullable [B, rows, D]
  uint32_t* err_word;         // nullable
  int64_t B, S, W, rows, record_stride, start, total, ratio;
  int64_t k0, nk;             // the records this call closes: k0 .. k0 + nk - 1
  int D, n_rope, kind, width;
  float rope_base[64];        // 160000^(-2i / n_rope) per RoPE pair, binary32
  void* ev_before;            // nullable measurement events around the record kernel
  void* ev_after;
};
size_t compress_smem_bytes(int ratio, int64_t D);
int launch_compress(const CompressArgs& a, cudaStream_t st);
int launch_pool_weight(const float* t, float* w, int64_t n, cudaStream_t st);

// ---- paged: write the new token into the pool -----------------------------------
struct PagedAppendArgs {
  void* k_pool;
  void* v_pool;
  const void* k_new;
  const void* v_new;
  const int32_t* block_table;
  const int32_t* ctx_len;
  int64_t B, Hkv, D, page_tokens, max_pages, num_pages;
  int esz;
  uint32_t* err_word;
};
int launch_paged_append(const PagedAppendArgs& a, cudaStream_t st);

}  // namespace sa
