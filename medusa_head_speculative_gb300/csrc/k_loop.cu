// Bookkeeping kernel of the steady-state decode loop: after each step, append the step's
// emitted tokens and kept-token count to the caller's ring buffers at the position held
// by a device step counter, then advance the counter (so a captured step can be replayed
// without any host-side index).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace medusa {

__global__ void __launch_bounds__(256) loop_append_kernel(const int32_t* __restrict__ tok,
                                                          const int32_t* __restrict__ n_acc, int B,
                                                          int W, int max_steps, long long* count,
                                                          int32_t* ring_tok, int32_t* ring_nacc) {
  pdl_trigger();
  pdl_wait();
  const long long c = *count;                 // read by every thread before thread 0 moves it
  const long slot = (long)(c % max_steps);
  for (int e = threadIdx.x; e < B * W; e += blockDim.x) ring_tok[slot * B * W + e] = tok[e];
  for (int b = threadIdx.x; b < B; b += blockDim.x) ring_nacc[slot * B + b] = n_acc[b];
  __syncthreads();
  if (threadIdx.x == 0) *count = c + 1;
}

cudaError_t launch_loop_append(const int32_t* tok, const int32_t* n_acc, int B, int W, int max_steps,
                               long long* count, int32_t* ring_tok, int32_t* ring_nacc,
                               cudaStream_t st) {
  return launch_kernel(loop_append_kernel, dim3(1), dim3(256), 0, st, 1, tok, n_acc, B, W, max_steps,
                       count, ring_tok, ring_nacc);
}

}  // namespace medusa
