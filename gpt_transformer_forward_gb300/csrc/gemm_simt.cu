// gemm_simt.cu -- fp32 CUDA-core GEMM for the GPT2_FP32 precision mode.
//
//   out[m, n] (op)= sum_k A[m, k] * W[n, k] + bias[n]
//
// A 64 x 64 output tile per 256-thread block, 4 x 4 outputs per thread,
// K staged through shared memory 16 at a time.  Each output is one fp32 FMA
// chain in increasing k, so the result carries only fp32 rounding; this is
// the reference-grade mode, not the fast one.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kT = 64, kK = 16;

template <int kEpi>
__global__ void __launch_bounds__(256) gemm_simt_kernel(float* __restrict__ out, const float* __restrict__ A,
                                                        const float* __restrict__ W,
                                                        const float* __restrict__ bias, int M, int N, int K) {
  __shared__ float As[kK][kT + 4];
  __shared__ float Ws[kK][kT + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kK) {
    // 64 rows x 16 k of A and of W: 1024 values each, 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + i * 256;
      const int r = idx / kK, kk = idx % kK;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
      Ws[kk][r] = (gn < N && gk < K) ? W[static_cast<size_t>(gn) * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        w[i] = Ws[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j] + (bias ? bias[n] : 0.f);
      float* o = out + static_cast<size_t>(m) * N + n;
      if constexpr (kEpi == kEpiGelu16) {
        v = gelu_exact(v);  // fp32 mode keeps an fp32 output
      }
      if constexpr (kEpi == kEpiResidF32) v = *o + v;
      *o = v;
    }
  }
}

}  // namespace

void launch_gemm_simt(float* out, const float* A, const float* W, const float* bias, int M, int N, int K, int epi,
                      cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT);
  switch (epi) {
    case kEpiGelu16: gemm_simt_kernel<kEpiGelu16><<<grid, 256, 0, s>>>(out, A, W, bias, M, N, K); break;
    case kEpiResidF32: gemm_simt_kernel<kEpiResidF32><<<grid, 256, 0, s>>>(out, A, W, bias, M, N, K); break;
    default: gemm_simt_kernel<kEpiF32><<<grid, 256, 0, s>>>(out, A, W, bias, M, N, K); break;
  }
}

}  // namespace gpt2
