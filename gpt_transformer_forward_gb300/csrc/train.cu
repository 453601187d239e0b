// train.cu -- the kernels of a GPT-2 training step beyond the forward pass
// (llm.c "State of the Union": the classifier's softmax cross-entropy, the
// backward blocks -- matmul backward with its bias, layernorm backward, gelu
// backward, attention backward, encoder backward -- and AdamW), fp32.
//
// The matmul backward products run on the GEMM kernels of the forward pass
// (fp32 CUDA cores, or tcgen05 with tf32 operands), which take both
// operands K-major: the transposes they need are made here.  Column sums
// (bias gradients, LayerNorm's weight gradients) are deterministic: partial
// sums over fixed row chunks, then one sum over the chunks in a fixed order.
// Only the token-embedding gradient of the encoder scatters with atomics
// (a token may repeat), so its low bits can change from run to run.
#include "kernels.cuh"

namespace gpt2 {
namespace {

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red may still be read from a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];  // every thread, the same order
  return s;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = -INFINITY;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  return m;
}

// out[c][r] = in[r][c] for a rows x cols matrix; 32 x 32 tiles through
// shared memory (padded), block 32 x 8
__global__ void transpose_kernel(float* __restrict__ out, const float* __restrict__ in, int rows, int cols) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = in[static_cast<size_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < rows) out[static_cast<size_t>(c) * rows + r] = tile[threadIdx.x][i];
  }
}

// Softmax cross-entropy of one row of logits over the first V columns, the
// row's loss -log p[target] into losses[n], and dlogits = (p - onehot) *
// inv_n written over the logits (0 in the padded columns).  A target
// outside [0, V) is flagged and read as 0.
__global__ void __launch_bounds__(512) crossentropy_kernel(float* __restrict__ logits, float* __restrict__ losses,
                                                           const int* __restrict__ targets, int V, int Vp,
                                                           float inv_n) {
  __shared__ float red[32];
  float* row = logits + static_cast<size_t>(blockIdx.x) * Vp;
  int tgt = targets[blockIdx.x];
  if (tgt < 0 || tgt >= V) {
    if (threadIdx.x == 0) set_error(GPT2_DEVERR_TOKEN);
    tgt = 0;
  }
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) mx = fmaxf(mx, row[v]);
  mx = block_max(mx, red);
  float sum = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) sum += expf(row[v] - mx);
  sum = block_sum(sum, red);
  const float lt = row[tgt];  // read by every thread before any writes below
  __syncthreads();
  if (threadIdx.x == 0) losses[blockIdx.x] = -(lt - mx - logf(sum));
  const float inv_sum = 1.0f / sum;
  for (int v = threadIdx.x; v < Vp; v += blockDim.x) {
    const float p = v < V ? expf(row[v] - mx) * inv_sum : 0.f;
    row[v] = (p - (v == tgt ? 1.f : 0.f)) * inv_n;
  }
}

// out[0] = mean of in[0 .. n): one block, a fixed summation order
__global__ void __launch_bounds__(1024) mean_kernel(float* __restrict__ out, const float* __restrict__ in, int n) {
  __shared__ float red[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += in[i];
  s = block_sum(s, red);
  if (threadIdx.x == 0) out[0] = s / static_cast<float>(n);
}

// part[p][c] = sum of in[r][c] over rows r in [p * rows_per_part, ...);
// grid (column blocks of 256, parts)
__global__ void column_partial_kernel(float* __restrict__ part, const float* __restrict__ in, int rows, int cols,
                                      int rows_per_part) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int r0 = blockIdx.y * rows_per_part, r1 = min(rows, r0 + rows_per_part);
  float s = 0.f;
  for (int r = r0; r < r1; ++r) s += in[static_cast<size_t>(r) * cols + c];
  part[static_cast<size_t>(blockIdx.y) * cols + c] = s;
}

// out[c] = (out[c] +) sum over the parts of part[p][c], in part order
__global__ void column_sum_kernel(float* __restrict__ out, const float* __restrict__ part, int parts, int cols,
                                  int accumulate) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float s = accumulate ? out[c] : 0.f;
  for (int p = 0; p < parts; ++p) s += part[static_cast<size_t>(p) * cols + c];
  out[c] = s;
}

// LayerNorm backward, one warp per row: with xhat = (x - mean) rstd and
// g = dy w, dx = rstd (g - mean_c(g) - xhat mean_c(g xhat)), accumulated
// into dx when accumulate (the residual stream's gradient)
__global__ void __launch_bounds__(256) layernorm_backward_dx_kernel(float* __restrict__ dx, const float* __restrict__ dy,
                                                                    const float* __restrict__ x,
                                                                    const float* __restrict__ w,
                                                                    const float* __restrict__ mean,
                                                                    const float* __restrict__ rstd, int N, int C,
                                                                    int accumulate) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= N) return;
  const float* dyr = dy + static_cast<size_t>(row) * C;
  const float* xr = x + static_cast<size_t>(row) * C;
  const float mu = mean[row], rs = rstd[row];
  float mg = 0.f, mgx = 0.f;
  for (int c = lane; c < C; c += 32) {
    const float g = dyr[c] * w[c];
    mg += g;
    mgx += g * (xr[c] - mu) * rs;
  }
  mg = warp_sum(mg) / C;
  mgx = warp_sum(mgx) / C;
  float* dxr = dx + static_cast<size_t>(row) * C;
  for (int c = lane; c < C; c += 32) {
    const float v = rs * (dyr[c] * w[c] - mg - (xr[c] - mu) * rs * mgx);
    dxr[c] = accumulate ? dxr[c] + v : v;
  }
}

// LayerNorm's weight and bias gradients, partial sums over row chunks:
// part_w[p][c] = sum dy xhat, part_b[p][c] = sum dy
__global__ void layernorm_backward_wb_kernel(float* __restrict__ part_w, float* __restrict__ part_b,
                                             const float* __restrict__ dy, const float* __restrict__ x,
                                             const float* __restrict__ mean, const float* __restrict__ rstd, int N,
                                             int C, int rows_per_part) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  const int r0 = blockIdx.y * rows_per_part, r1 = min(N, r0 + rows_per_part);
  float sw = 0.f, sb = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float d = dy[static_cast<size_t>(r) * C + c];
    sw += d * (x[static_cast<size_t>(r) * C + c] - mean[r]) * rstd[r];
    sb += d;
  }
  part_w[static_cast<size_t>(blockIdx.y) * C + c] = sw;
  part_b[static_cast<size_t>(blockIdx.y) * C + c] = sb;
}

// dinp = dout * GELU'(inp), GELU in the tanh form
__global__ void gelu_backward_kernel(float* __restrict__ dinp, const float* __restrict__ inp,
                                     const float* __restrict__ dout, long long n) {
  const float k = 0.7978845608028654f;  // sqrt(2/pi)
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float x = inp[i];
    const float th = tanhf(k * (x + 0.044715f * x * x * x));
    const float d = 0.5f * (1.f + th) + 0.5f * x * (1.f - th * th) * k * (1.f + 3.f * 0.044715f * x * x);
    dinp[i] = dout[i] * d;
  }
}

// dwpe[t][c] = sum over sequences of dx[b][t][c] (positions < T)
__global__ void encoder_backward_wpe_kernel(float* __restrict__ dwpe, const float* __restrict__ dx, int B, int T,
                                            int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * C) return;
  float s = 0.f;
  for (int b = 0; b < B; ++b) s += dx[static_cast<size_t>(b) * T * C + i];
  dwpe[i] = s;
}

// dwte[tok[n]][c] += dx[n][c] (tokens may repeat: atomics)
__global__ void encoder_backward_wte_kernel(float* __restrict__ dwte, const float* __restrict__ dx,
                                            const int* __restrict__ tok, int N, int C, int V) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= static_cast<long long>(N) * C) return;
  const int n = static_cast<int>(i / C), c = static_cast<int>(i % C);
  int ix = tok[n];
  if (ix < 0 || ix >= V) return;  // flagged by the forward's encoder
  atomicAdd(dwte + static_cast<size_t>(ix) * C + c, dx[i]);
}

// AdamW: m = b1 m + (1 - b1) g, v = b2 v + (1 - b2) g^2,
// p -= lr (m / c1 / (sqrt(v / c2) + eps) + wd p), c1 = 1 - b1^t, c2 = 1 - b2^t
__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                             float* __restrict__ v, long long n, float lr, float b1, float b2, float eps, float wd,
                             float c1, float c2) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float gi = g[i];
    const float mi = b1 * m[i] + (1.f - b1) * gi;
    const float vi = b2 * v[i] + (1.f - b2) * gi * gi;
    m[i] = mi;
    v[i] = vi;
    p[i] -= lr * ((mi / c1) / (sqrtf(vi / c2) + eps) + wd * p[i]);
  }
}

unsigned grid_for(long long n, int threads) {
  const long long cap = static_cast<long long>(num_sms()) * 16;
  const long long want = (n + threads - 1) / threads;
  return static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
}

constexpr int kPartRows = 256;  // rows per partial sum of a column reduction

}  // namespace

int column_parts(int rows) { return (rows + kPartRows - 1) / kPartRows; }

void launch_transpose(float* out, const float* in, int rows, int cols, cudaStream_t s) {
  transpose_kernel<<<dim3((cols + 31) / 32, (rows + 31) / 32), dim3(32, 8), 0, s>>>(out, in, rows, cols);
}

void launch_crossentropy(float* logits, float* losses, float* loss, const int* targets, int N, int V, int Vp,
                         cudaStream_t s) {
  crossentropy_kernel<<<N, 512, 0, s>>>(logits, losses, targets, V, Vp, 1.0f / static_cast<float>(N));
  mean_kernel<<<1, 1024, 0, s>>>(loss, losses, N);
}

void launch_column_sum(float* out, float* part, const float* in, int rows, int cols, bool accumulate, cudaStream_t s) {
  const int parts = column_parts(rows);
  column_partial_kernel<<<dim3((cols + 255) / 256, parts), 256, 0, s>>>(part, in, rows, cols, kPartRows);
  column_sum_kernel<<<(cols + 255) / 256, 256, 0, s>>>(out, part, parts, cols, accumulate ? 1 : 0);
}

void launch_layernorm_backward(float* dx, float* dw, float* db, float* part, const float* dy, const float* x,
                               const float* w, const float* mean, const float* rstd, int N, int C, bool accumulate,
                               cudaStream_t s) {
  layernorm_backward_dx_kernel<<<(N + 7) / 8, 256, 0, s>>>(dx, dy, x, w, mean, rstd, N, C, accumulate ? 1 : 0);
  const int parts = column_parts(N);
  float* part_w = part;
  float* part_b = part + static_cast<size_t>(parts) * C;
  layernorm_backward_wb_kernel<<<dim3((C + 255) / 256, parts), 256, 0, s>>>(part_w, part_b, dy, x, mean, rstd, N, C,
                                                                            kPartRows);
  column_sum_kernel<<<(C + 255) / 256, 256, 0, s>>>(dw, part_w, parts, C, 0);
  column_sum_kernel<<<(C + 255) / 256, 256, 0, s>>>(db, part_b, parts, C, 0);
}

void launch_gelu_backward(float* dinp, const float* inp, const float* dout, long long n, cudaStream_t s) {
  gelu_backward_kernel<<<grid_for(n, 256), 256, 0, s>>>(dinp, inp, dout, n);
}

void launch_encoder_backward(float* dwte, float* dwpe, const float* dx, const int* tok, int B, int T, int C, int V,
                             cudaStream_t s) {
  encoder_backward_wpe_kernel<<<(T * C + 255) / 256, 256, 0, s>>>(dwpe, dx, B, T, C);
  const long long n = static_cast<long long>(B) * T * C;
  encoder_backward_wte_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(dwte, dx, tok, B * T, C, V);
}

void launch_adamw(float* p, const float* g, float* m, float* v, long long n, float lr, float b1, float b2, float eps,
                  float wd, int t, cudaStream_t s) {
  const float c1 = 1.f - powf(b1, static_cast<float>(t)), c2 = 1.f - powf(b2, static_cast<float>(t));
  adamw_kernel<<<grid_for(n, 256), 256, 0, s>>>(p, g, m, v, n, lr, b1, b2, eps, wd, c1, c2);
}

}  // namespace gpt2
