// noalloc.cu -- matmul_forward for callers that cannot allocate device memory.
//
// matmul_forward's 16-bit tensor-core modes need scratch space for the
// 16-bit copies of `inp` and `W`, which the caller normally passes in as a
// workspace.  Some callers have no way to get one: code that must never call
// cudaMalloc (it can synchronise the device and stall other work), plugins
// loaded into a host program that owns every device allocation and offers no
// workspace, or programs with a fixed device-memory budget.  For them this
// file keeps the scratch in a fixed device array that is part of the library
// image: every GPU that loads the library holds these bytes until the
// process exits.
#include <mutex>

#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

// The scratch itself.  In host code this name is only a stand-in for the
// device object; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_matmul_scratch[kNoAllocScratchBytes];

// Device address of g_matmul_scratch, looked up once per device (with that
// device current) on the first call made on it.
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_matmul_scratch);
    if (e != cudaSuccess) return note_cuda_error(e);  // keeps the error text for gpt2_last_cuda_error()
    if (p == nullptr) return GPT2_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return GPT2_OK;
}

}  // namespace
}  // namespace gpt2

extern "C" int matmul_forward_noalloc(float* out, const float* inp, const float* W, const float* bias, int N, int C,
                                      int OC, int precision, void* stream) {
  const size_t need = matmul_workspace_size(N, C, OC, precision);
  if (need > gpt2::kNoAllocScratchBytes) return GPT2_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = gpt2::scratch_address(&scratch);
    if (rc != GPT2_OK) return rc;
  }
  // Every call overwrites the scratch before reading it, so nothing in it
  // has to start at zero.
  return matmul_forward(out, inp, W, bias, N, C, OC, precision, scratch, need, stream);
}
