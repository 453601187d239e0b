// diag.cu -- a check of the library's bounded-wait path on the device.
//
// Every pipeline wait in the kernels (an mbarrier phase that TMA copies or
// tensor-core commits complete) gives up after a time limit instead of
// spinning forever: it sets GPT2_DEVERR_TIMEOUT in the device error word and
// the kernel winds down and returns.  gpt2_diag_wait_timeout() runs that
// path on purpose: one CTA initialises an mbarrier that no thread or copy
// ever arrives at and waits on it with the same wait function and a short
// limit, so that a test can see the wait end, the error bit set and the
// device stay usable for the next call.
#include "kernels.cuh"

namespace gpt2 {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned long long limit_ns, int* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1u);  // one arrival expected; none comes
    fence_barrier_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0u, limit_ns);
  if (threadIdx.x == 0) *gave_up = ok ? 0 : 1;
}

}  // namespace
}  // namespace gpt2

extern "C" int gpt2_diag_wait_timeout(long long limit_ns, int* gave_up, void* stream) {
  if (gave_up == nullptr || limit_ns < 1000 || limit_ns > 1000000000LL) return GPT2_ERR_ARG;
  gpt2::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(limit_ns), gave_up);
  const cudaError_t e = cudaPeekAtLastError();
  return e == cudaSuccess ? GPT2_OK : gpt2::note_cuda_error(e);
}
