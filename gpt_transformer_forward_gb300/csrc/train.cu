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

// out[c][r] = in[r][c] for a rows x cols matrix: 64 x 64 tiles through
// shared memory (rows padded to 65 words), 256 threads (16 x 16).  With vec
// (rows and cols multiples of 4, 16-byte aligned pointers) a full tile moves
// as 16-byte loads along the rows of in and 16-byte stores along the rows of
// out (measured: the 32 x 32 tile with 4-byte accesses moved 2.9 TB/s);
// edge tiles take guarded 4-byte accesses.
__global__ void __launch_bounds__(256) transpose_kernel(float* __restrict__ out, const float* __restrict__ in,
                                                        int rows, int cols, int vec) {
  __shared__ float tile[64][65];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool full = vec && r0 + 64 <= rows && c0 + 64 <= cols;
  if (full) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // rows r0 + ty + 16 k, columns c0 + 4 tx .. + 3
      const float4 v = __ldg(reinterpret_cast<const float4*>(in + static_cast<size_t>(r0 + ty + 16 * k) * cols + c0) + tx);
      float* t = &tile[ty + 16 * k][4 * tx];
      t[0] = v.x;
      t[1] = v.y;
      t[2] = v.z;
      t[3] = v.w;
    }
  } else {
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
      const int r = i >> 6, c = i & 63;
      if (r0 + r < rows && c0 + c < cols) tile[r][c] = in[static_cast<size_t>(r0 + r) * cols + c0 + c];
    }
  }
  __syncthreads();
  if (full) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // out rows c0 + ty + 16 k, columns r0 + 4 tx .. + 3
      const int c = ty + 16 * k;
      const float4 v = make_float4(tile[4 * tx][c], tile[4 * tx + 1][c], tile[4 * tx + 2][c], tile[4 * tx + 3][c]);
      reinterpret_cast<float4*>(out + static_cast<size_t>(c0 + c) * rows + r0)[tx] = v;
    }
  } else {
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
      const int c = i >> 6, r = i & 63;
      if (c0 + c < cols && r0 + r < rows) out[static_cast<size_t>(c0 + c) * rows + r0 + r] = tile[r][c];
    }
  }
}

// Softmax cross-entropy of one row of logits over the first V columns, the
// row's loss -log p[target] into losses[n], and dlogits = (p - onehot) *
// inv_n written over the logits (0 in the padded columns).  A target
// outside [0, V) is flagged and read as 0.  One block per row: a first
// pass keeps a running (maximum, sum of exponentials) per thread over
// 16-byte loads (vec: Vp a multiple of 4), merged over the block; a second
// pass, whose reads of the row mostly hit L2, writes the gradient.  The
// exponentials are exp2 of x log2(e) - max log2(e) on the SFU.
constexpr int kCeThreads = 1024;
__global__ void __launch_bounds__(kCeThreads) crossentropy_kernel(float* __restrict__ logits,
                                                                  float* __restrict__ losses,
                                                                  const int* __restrict__ targets, int V, int Vp,
                                                                  float inv_n, int vec) {
  __shared__ float red[32];
  constexpr float kLog2e = 1.4426950408889634f;
  float* row = logits + static_cast<size_t>(blockIdx.x) * Vp;
  int tgt = targets[blockIdx.x];
  if (tgt < 0 || tgt >= V) {
    if (threadIdx.x == 0) set_error(GPT2_DEVERR_TOKEN);
    tgt = 0;
  }
  float mx = -INFINITY, sum = 0.f;  // this thread's running maximum and sum of exp(x - mx)
  auto take = [&](float a, float b, float c, float d) {
    const float m4 = fmaxf(fmaxf(a, b), fmaxf(c, d));
    if (m4 == -INFINITY) return;
    const float m_new = fmaxf(mx, m4), nb = -m_new * kLog2e;
    sum = sum * exp2_approx(fmaf(mx, kLog2e, nb)) + exp2_approx(fmaf(a, kLog2e, nb)) +
          exp2_approx(fmaf(b, kLog2e, nb)) + exp2_approx(fmaf(c, kLog2e, nb)) + exp2_approx(fmaf(d, kLog2e, nb));
    mx = m_new;
  };
  if (vec) {
    for (int v = 4 * threadIdx.x; v < V; v += 4 * kCeThreads) {
      const float4 x = *reinterpret_cast<const float4*>(row + v);
      take(x.x, v + 1 < V ? x.y : -INFINITY, v + 2 < V ? x.z : -INFINITY, v + 3 < V ? x.w : -INFINITY);
    }
  } else {
    for (int v = threadIdx.x; v < V; v += kCeThreads) take(row[v], -INFINITY, -INFINITY, -INFINITY);
  }
  const float m_row = block_max(mx, red);
  sum = block_sum(mx == -INFINITY ? 0.f : sum * exp2_approx((mx - m_row) * kLog2e), red);
  const float lt = row[tgt];  // read by every thread before any writes below
  __syncthreads();
  if (threadIdx.x == 0) losses[blockIdx.x] = -(lt - m_row - logf(sum));
  const float scale = inv_n / sum, nb = -m_row * kLog2e;
  if (vec) {
    for (int v = 4 * threadIdx.x; v < Vp; v += 4 * kCeThreads) {
      float4 x = *reinterpret_cast<const float4*>(row + v);
      x.x = v < V ? exp2_approx(fmaf(x.x, kLog2e, nb)) * scale : 0.f;
      x.y = v + 1 < V ? exp2_approx(fmaf(x.y, kLog2e, nb)) * scale : 0.f;
      x.z = v + 2 < V ? exp2_approx(fmaf(x.z, kLog2e, nb)) * scale : 0.f;
      x.w = v + 3 < V ? exp2_approx(fmaf(x.w, kLog2e, nb)) * scale : 0.f;
      if (tgt >= v && tgt < v + 4) {
        const int k = tgt - v;
        if (k == 0) x.x -= inv_n;
        if (k == 1) x.y -= inv_n;
        if (k == 2) x.z -= inv_n;
        if (k == 3) x.w -= inv_n;
      }
      *reinterpret_cast<float4*>(row + v) = x;
    }
  } else {
    for (int v = threadIdx.x; v < Vp; v += kCeThreads) {
      const float p = v < V ? exp2_approx(fmaf(row[v], kLog2e, nb)) * scale : 0.f;
      row[v] = p - (v == tgt ? inv_n : 0.f);
    }
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
                                      int rows_per_part, int vec) {
  const int r0 = blockIdx.y * rows_per_part, r1 = min(rows, r0 + rows_per_part);
  if (vec) {  // four columns per thread, 16-byte loads
    const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (c >= cols) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(in + static_cast<size_t>(r) * cols + c));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<float4*>(part + static_cast<size_t>(blockIdx.y) * cols + c) = acc;
  } else {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    float acc = 0.f;
    for (int r = r0; r < r1; ++r) acc += in[static_cast<size_t>(r) * cols + c];
    part[static_cast<size_t>(blockIdx.y) * cols + c] = acc;
  }
}

// out[c] = (out[c] +) sum over the parts of part[p][c].  A block of 256
// threads takes 32 columns: warp g sums parts g, g + 8, ... of its lane's
// column in part order (each warp load one 128-byte row piece), and the
// eight sums are added in warp order, a fixed order, so the result does
// not depend on timing.  (One thread per column, adding all its parts in
// turn, left a 768-column reduction 3 blocks for the whole GPU: about 20 us
// per launch, measured.)
constexpr int kColSumCols = 32;
constexpr int kColSumGroups = 8;
__global__ void __launch_bounds__(kColSumCols* kColSumGroups)
    column_sum_kernel(float* __restrict__ out, const float* __restrict__ part, int parts, int cols, int accumulate) {
  __shared__ float red[kColSumGroups][kColSumCols + 1];
  const int cl = threadIdx.x % kColSumCols, g = threadIdx.x / kColSumCols;
  const int c = blockIdx.x * kColSumCols + cl;
  float s = 0.f;
  if (c < cols) {
#pragma unroll 4
    for (int p = g; p < parts; p += kColSumGroups) s += __ldg(part + static_cast<size_t>(p) * cols + c);
  }
  red[g][cl] = s;
  __syncthreads();
  if (g == 0 && c < cols) {
    float t = accumulate ? out[c] : 0.f;
#pragma unroll
    for (int k = 0; k < kColSumGroups; ++k) t += red[k][cl];
    out[c] = t;
  }
}

void launch_column_sum_parts(float* out, const float* part, int parts, int cols, bool accumulate, cudaStream_t s) {
  column_sum_kernel<<<(cols + kColSumCols - 1) / kColSumCols, kColSumCols * kColSumGroups, 0, s>>>(
      out, part, parts, cols, accumulate ? 1 : 0);
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
                                             int C, int rows_per_part, int vec) {
  const int r0 = blockIdx.y * rows_per_part, r1 = min(N, r0 + rows_per_part);
  if (vec) {  // four columns per thread, 16-byte loads
    const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (c >= C) return;
    float4 sw = make_float4(0.f, 0.f, 0.f, 0.f), sb = sw;
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      const size_t at = static_cast<size_t>(r) * C + c;
      const float4 d = __ldg(reinterpret_cast<const float4*>(dy + at));
      const float4 xv = __ldg(reinterpret_cast<const float4*>(x + at));
      const float mr = __ldg(mean + r), rr = __ldg(rstd + r);
      sw.x += d.x * (xv.x - mr) * rr;
      sw.y += d.y * (xv.y - mr) * rr;
      sw.z += d.z * (xv.z - mr) * rr;
      sw.w += d.w * (xv.w - mr) * rr;
      sb.x += d.x;
      sb.y += d.y;
      sb.z += d.z;
      sb.w += d.w;
    }
    *reinterpret_cast<float4*>(part_w + static_cast<size_t>(blockIdx.y) * C + c) = sw;
    *reinterpret_cast<float4*>(part_b + static_cast<size_t>(blockIdx.y) * C + c) = sb;
  } else {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float sw = 0.f, sb = 0.f;
    for (int r = r0; r < r1; ++r) {
      const float d = dy[static_cast<size_t>(r) * C + c];
      sw += d * (x[static_cast<size_t>(r) * C + c] - mean[r]) * rstd[r];
      sb += d;
    }
    part_w[static_cast<size_t>(blockIdx.y) * C + c] = sw;
    part_b[static_cast<size_t>(blockIdx.y) * C + c] = sb;
  }
}

// dinp = dout * GELU'(inp), GELU in the tanh form
__global__ void gelu_backward_kernel(float* __restrict__ dinp, const float* __restrict__ inp,
                                     const float* __restrict__ dout, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dinp[i] = dout[i] * gelu_grad(inp[i]);
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
__device__ __forceinline__ void adamw_one(float& p, float g, float& m, float& v, float lr, float b1, float b2,
                                          float eps, float wd, float c1, float c2) {
  m = b1 * m + (1.f - b1) * g;
  v = b2 * v + (1.f - b2) * g * g;
  p -= lr * ((m / c1) / (sqrtf(v / c2) + eps) + wd * p);
}

// vec (the four buffers 16-byte aligned): four parameters per iteration
// with 16-byte accesses, then the tail of n % 4; else one at a time
__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                             float* __restrict__ v, long long n, float lr, float b1, float b2, float eps, float wd,
                             float c1, float c2, int vec) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (!vec) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride)
      adamw_one(p[i], g[i], m[i], v[i], lr, b1, b2, eps, wd, c1, c2);
    return;
  }
  const long long n4 = n / 4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4; i += stride) {
    float4 pi = reinterpret_cast<float4*>(p)[i], mi = reinterpret_cast<float4*>(m)[i],
           vi = reinterpret_cast<float4*>(v)[i];
    const float4 gi = __ldg(reinterpret_cast<const float4*>(g) + i);
    adamw_one(pi.x, gi.x, mi.x, vi.x, lr, b1, b2, eps, wd, c1, c2);
    adamw_one(pi.y, gi.y, mi.y, vi.y, lr, b1, b2, eps, wd, c1, c2);
    adamw_one(pi.z, gi.z, mi.z, vi.z, lr, b1, b2, eps, wd, c1, c2);
    adamw_one(pi.w, gi.w, mi.w, vi.w, lr, b1, b2, eps, wd, c1, c2);
    reinterpret_cast<float4*>(p)[i] = pi;
    reinterpret_cast<float4*>(m)[i] = mi;
    reinterpret_cast<float4*>(v)[i] = vi;
  }
  if (blockIdx.x == 0 && threadIdx.x < n - 4 * n4) {
    const long long i = 4 * n4 + threadIdx.x;
    adamw_one(p[i], g[i], m[i], v[i], lr, b1, b2, eps, wd, c1, c2);
  }
}

unsigned grid_for(long long n, int threads) {
  const long long cap = static_cast<long long>(num_sms()) * 16;
  const long long want = (n + threads - 1) / threads;
  return static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
}

constexpr int kPartRows = 64;  // rows per partial sum of a column reduction

}  // namespace

int column_parts(int rows) { return (rows + kPartRows - 1) / kPartRows; }

void launch_transpose(float* out, const float* in, int rows, int cols, cudaStream_t s) {
  const int vec = (rows % 4 == 0 && cols % 4 == 0 && (reinterpret_cast<uintptr_t>(in) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15u) == 0)
                      ? 1
                      : 0;
  transpose_kernel<<<dim3((cols + 63) / 64, (rows + 63) / 64), 256, 0, s>>>(out, in, rows, cols, vec);
}

void launch_crossentropy(float* logits, float* losses, float* loss, const int* targets, int N, int V, int Vp,
                         cudaStream_t s) {
  const int vec = (Vp % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) ? 1 : 0;
  crossentropy_kernel<<<N, kCeThreads, 0, s>>>(logits, losses, targets, V, Vp, 1.0f / static_cast<float>(N), vec);
  mean_kernel<<<1, 1024, 0, s>>>(loss, losses, N);
}

void launch_column_sum(float* out, float* part, const float* in, int rows, int cols, bool accumulate, cudaStream_t s) {
  const int parts = column_parts(rows);
  const int vec = (cols % 4 == 0 && (reinterpret_cast<uintptr_t>(in) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(part) & 15u) == 0)
                      ? 1
                      : 0;
  const int per_block = vec ? 1024 : 256;  // columns per block of 256 threads
  column_partial_kernel<<<dim3((cols + per_block - 1) / per_block, parts), 256, 0, s>>>(part, in, rows, cols,
                                                                                       kPartRows, vec);
  launch_column_sum_parts(out, part, parts, cols, accumulate, s);
}

void launch_layernorm_backward(float* dx, float* dw, float* db, float* part, const float* dy, const float* x,
                               const float* w, const float* mean, const float* rstd, int N, int C, bool accumulate,
                               cudaStream_t s) {
  layernorm_backward_dx_kernel<<<(N + 7) / 8, 256, 0, s>>>(dx, dy, x, w, mean, rstd, N, C, accumulate ? 1 : 0);
  const int parts = column_parts(N);
  float* part_w = part;
  float* part_b = part + static_cast<size_t>(parts) * C;
  const int vec = (C % 4 == 0 && (reinterpret_cast<uintptr_t>(dy) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(part) & 15u) == 0)
                      ? 1
                      : 0;
  const int per_block = vec ? 1024 : 256;
  layernorm_backward_wb_kernel<<<dim3((C + per_block - 1) / per_block, parts), 256, 0, s>>>(
      part_w, part_b, dy, x, mean, rstd, N, C, kPartRows, vec);
  launch_column_sum_parts(dw, part_w, parts, C, false, s);
  launch_column_sum_parts(db, part_b, parts, C, false, s);
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
  const int vec = ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(m) |
                    reinterpret_cast<uintptr_t>(v)) &
                   15u) == 0
                      ? 1
                      : 0;
  adamw_kernel<<<grid_for(vec ? n / 4 + 1 : n, 256), 256, 0, s>>>(p, g, m, v, n, lr, b1, b2, eps, wd, c1, c2, vec);
}

}  // namespace gpt2
