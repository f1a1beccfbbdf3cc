// k_diag.cu -- the bounded-wait timeout path, run on purpose and without a fault.
//
// Every pipelined kernel of the library waits on mbarriers through
// wait_or_abort / mbar_wait, which give up after kWaitCycles SM cycles, OR
// SA_ERRBIT_TIMEOUT into the caller's error word and let the CTA return.  That
// path only runs when a producer never arrives, which a correct call never
// causes; this kernel makes it run: one warp waits on a barrier that nothing
// arrives on (no copy or MMA is in flight), then checks that a second wait in
// the same CTA returns at once on the abort flag the first one set.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace sa {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t* err_word, uint32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // count 1; nothing ever arrives
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  volatile int* ab = &abort_flag;
  const long long t0 = clock64();
  const bool first = wait_or_abort(&bar, 0, ab, err_word);  // runs out
  const long long t1 = clock64();
  const bool second = wait_or_abort(&bar, 0, ab, err_word);  // abort flag already set
  const long long t2 = clock64();
  // out[0]: 1 if the first wait gave up; out[1]: 1 if the second returned
  // false within 2^20 cycles; out[2], out[3]: the first wait's cycles (lo, hi)
  out[0] = first ? 0u : 1u;
  out[1] = (!second && t2 - t1 < (1LL << 20)) ? 1u : 0u;
  out[2] = static_cast<uint32_t>(t1 - t0);
  out[3] = static_cast<uint32_t>((t1 - t0) >> 32);
}

int launch_wait_timeout(uint32_t* err_word, uint32_t* out, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err_word, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
