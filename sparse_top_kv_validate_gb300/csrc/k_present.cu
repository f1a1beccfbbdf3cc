// k_present.cu -- present K/V construction (past ++ current), a pure copy.
//
// Semantics: IndexShare `build_present` and ONNX Attention `build_kv`
// (onnx-runtime-ep-cuda src/kernels/index_share.rs, standard_attention.rs):
// present[b,h,t] = past[b,h,t] for t < P, cur[b,h,t-P] after; the capacity
// form writes the current token(s) at a per-batch position of a fixed-stride
// cache.
//
// GB300 mapping: every (b, h, t) row of D elements is moved with 16-byte
// vector loads/stores when the row size allows, K and V in one launch
// (blockIdx.y).  Only the rows that change are touched: in-place append
// writes C rows per (b, h) instead of rebuilding the cache.
#include "common.cuh"
#include "kernels.h"

namespace sa {

template <typename V>
__global__ void __launch_bounds__(256) present_kernel(PresentArgs a) {
  const int tsel = blockIdx.y;
  const char* past = static_cast<const char*>(a.past[tsel]);
  const char* cur = static_cast<const char*>(a.cur[tsel]);
  char* out = static_cast<char*>(a.present[tsel]);
  const int64_t row_vecs = a.D * a.esz / static_cast<int64_t>(sizeof(V));
  const int64_t row_bytes = a.D * a.esz;
  // positions handled per (b, h)
  int64_t span;
  if (a.write_pos == nullptr) span = a.P + a.C;          // concat
  else if (a.copy_past) span = a.stride;                 // full copy + append
  else span = a.C;                                       // in-place append
  const int64_t total = a.B * a.H * span * row_vecs;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t vi = e % row_vecs;
    int64_t r = e / row_vecs;
    const int64_t s = r % span;
    r /= span;
    const int64_t h = r % a.H;
    const int64_t b = r / a.H;
    const int64_t bh = b * a.H + h;
    const char* src;
    int64_t t;
    if (a.write_pos == nullptr) {
      t = s;
      src = (t < a.P) ? past + (bh * a.P + t) * row_bytes
                      : cur + (bh * a.C + (t - a.P)) * row_bytes;
    } else {
      const int64_t wp = a.write_pos[b];
      const bool ok = wp >= 0 && wp <= a.stride - a.C;
      if (!ok) {
        if (vi == 0 && s == 0 && h == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_WRITE_POS);
        continue;
      }
      if (a.copy_past) {
        t = s;
        src = (t >= wp && t < wp + a.C) ? cur + (bh * a.C + (t - wp)) * row_bytes
                                        : past + (bh * a.stride + t) * row_bytes;
      } else {
        t = wp + s;
        src = cur + (bh * a.C + s) * row_bytes;
      }
    }
    const V* sv = reinterpret_cast<const V*>(src) + vi;
    V* dv = reinterpret_cast<V*>(out + (bh * a.stride + t) * row_bytes) + vi;
    *dv = *sv;
  }
}

int launch_present(const PresentArgs& a, cudaStream_t st) {
  int64_t span = a.write_pos == nullptr ? a.P + a.C : (a.copy_past ? a.stride : a.C);
  const int64_t row_bytes = a.D * a.esz;
  bool vec16 = (row_bytes % 16) == 0;
  for (int i = 0; i < a.n_tensors && vec16; ++i) {
    vec16 = ((reinterpret_cast<uintptr_t>(a.present[i]) | reinterpret_cast<uintptr_t>(a.cur[i]) |
              reinterpret_cast<uintptr_t>(a.past[i])) & 15) == 0;
  }
  const int64_t vsz = vec16 ? 16 : a.esz;
  const int64_t total = a.B * a.H * span * (row_bytes / vsz);
  if (total == 0) return 0;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = 152 * 16;  // grid-stride beyond ~16 blocks per SM
  if (blocks > cap) blocks = cap;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(a.n_tensors));
  if (vec16) present_kernel<int4><<<grid, 256, 0, st>>>(a);
  else if (a.esz == 4) present_kernel<uint32_t><<<grid, 256, 0, st>>>(a);
  else present_kernel<uint16_t><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
