// pe_latency_floor: what a launch costs with (almost) no work in it, the
// reference against which the fused step is measured at small batch, where
// its time is mostly a chain of dependent round trips rather than bytes.
// A grid of `ctas` CTAs of 256 threads starts and ends; CTA 0's thread 0
// also follows `hops` dependent 4-byte loads through `chain` (entry i holds
// the index of the next entry) and stores where it ends.
#include "pe_internal.cuh"

namespace pe {

__global__ void __launch_bounds__(kThreads) floor_kernel(const int32_t* chain, int n, int hops,
                                                         int32_t* out) {
  if (blockIdx.x != 0 || threadIdx.x != 0 || hops == 0) return;
  int i = 0;
  for (int h = 0; h < hops; ++h) {
    i = __ldcg(chain + i);
    if ((unsigned)i >= (unsigned)n) i = 0;  // stay inside the chain
  }
  *out = i;
}

}  // namespace pe

extern "C" int pe_latency_floor(int32_t ctas, int32_t hops, const int32_t* chain, int32_t n,
                                int32_t* out, void* stream) {
  if (ctas < 1 || hops < 0 || (hops > 0 && (!chain || n < 1 || !out))) return PE_EINVAL;
  pe::floor_kernel<<<ctas, pe::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(chain, n, hops,
                                                                              out);
  return pe_host::launch_status();
}
