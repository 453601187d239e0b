// rowwise.cu -- the HBM-bound steps of the GPT-2 forward pass: encoder,
// LayerNorm, GELU, residual add, vocabulary softmax, argmax, plus the fp32
// to 16-bit (bf16 or fp16) conversions and the KV-cache writes the forward pass needs.
//
// Every kernel streams its rows with 128-bit loads and stores where the
// layout allows; row reductions are warp-shuffle (LayerNorm: one warp per
// row, the row held in registers) or block-wide (softmax: one block per
// row).
#include "kernels.cuh"

namespace gpt2 {

__device__ unsigned int g_error_word = 0;

// ---------------------------------------------------------------- encoder
// out[n, :] = wte[tok[n], :] + wpe[n % T, :], one float4 per thread.
// One warp per row: the token id is loaded once, then the row's wte and
// wpe float4s all in flight together (a thread per float4, each behind its
// own dependent token load, moved 3.3 TB/s: measured).
__global__ void __launch_bounds__(256) encoder_kernel(float4* __restrict__ out, const int* __restrict__ tok,
                                                      const float4* __restrict__ wte, const float4* __restrict__ wpe,
                                                      int N, int T, int C4, int V) {
  pdl_wait();  // x may still be read by the kernel ahead (the previous pass)
  pdl_trigger();
  const int n = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  int ix = __ldg(tok + n);
  if (ix < 0 || ix >= V) {
    if (lane == 0) set_error(GPT2_DEVERR_TOKEN);
    ix = 0;
  }
  const float4* a = wte + static_cast<size_t>(ix) * C4;
  const float4* p = wpe + static_cast<size_t>(n % T) * C4;
  float4* o = out + static_cast<size_t>(n) * C4;
  constexpr int kPer = 8;  // float4 per lane in flight
  for (int c0 = 0; c0 < C4; c0 += 32 * kPer) {
    float4 x[kPer], y[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int c = c0 + 32 * k + lane;
      if (c < C4) {
        x[k] = __ldg(a + c);
        y[k] = __ldg(p + c);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int c = c0 + 32 * k + lane;
      if (c < C4) o[c] = make_float4(x[k].x + y[k].x, x[k].y + y[k].y, x[k].z + y[k].z, x[k].w + y[k].w);
    }
  }
}

// Decode-step encoder: row b is token tok[b] at position pos (or pos_arr[b]).
__global__ void encoder_pos_kernel(float4* __restrict__ out, const int* __restrict__ tok,
                                   const float4* __restrict__ wte, const float4* __restrict__ wpe, int B, int pos_all,
                                   const int* __restrict__ pos_arr, int maxT, int C4, int V) {
  pdl_wait();  // tok comes from the argmax before it
  pdl_trigger();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * C4) return;
  const int b = idx / C4, c = idx % C4;
  int ix = __ldg(tok + b);
  if (ix < 0 || ix >= V) {
    if (c == 0) set_error(GPT2_DEVERR_TOKEN);
    ix = 0;
  }
  int pos = pos_arr != nullptr ? __ldg(pos_arr + b) : pos_all;
  if (pos < 0 || pos >= maxT) {
    if (c == 0) set_error(GPT2_DEVERR_POSITION);
    pos = 0;
  }
  const float4 a = __ldg(wte + static_cast<size_t>(ix) * C4 + c);
  const float4 p = __ldg(wpe + static_cast<size_t>(pos) * C4 + c);
  out[idx] = make_float4(a.x + p.x, a.y + p.y, a.z + p.z, a.w + p.w);
}

void launch_encoder(float* out, const int* tok, const float* wte, const float* wpe, int N, int T, int C, int V,
                    cudaStream_t s) {
  const int C4 = C / 4;
  const unsigned blocks = static_cast<unsigned>((N + 7) / 8);  // a warp per row
  launch_pdl(encoder_kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<float4*>(out), tok,
             reinterpret_cast<const float4*>(wte), reinterpret_cast<const float4*>(wpe), N, T, C4, V);
}

void launch_encoder_pos(float* out, const int* tok, const float* wte, const float* wpe, int B, int pos,
                        const int* pos_arr, int maxT, int C, int V, cudaStream_t s) {
  const int C4 = C / 4;
  const int threads = 256;
  launch_pdl(encoder_pos_kernel, dim3((B * C4 + threads - 1) / threads), dim3(threads), 0, s,
             reinterpret_cast<float4*>(out), tok, reinterpret_cast<const float4*>(wte),
             reinterpret_cast<const float4*>(wpe), B, pos, pos_arr, maxT, C4, V);
}

// -------------------------------------------------------------- LayerNorm
// One warp per row; the row's C = 128 * kVec floats sit in registers (kVec
// float4 per lane), so the mean and the variance of the centred values are
// two register passes over a single read.  Output fp32 or bf16.
template <int kVec, typename OutT>
__global__ void __launch_bounds__(256) layernorm_warp_kernel(OutT* __restrict__ out, float* __restrict__ mean_out,
                                                             float* __restrict__ rstd_out,
                                                             const float* __restrict__ inp,
                                                             const float* __restrict__ w,
                                                             const float* __restrict__ b, int N) {
  pdl_wait();
  pdl_trigger();
  constexpr int C = 128 * kVec;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= N) return;
  const float4* x4 = reinterpret_cast<const float4*>(inp + static_cast<size_t>(row) * C);
  float4 v[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) v[i] = __ldcs(x4 + lane + 32 * i);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  const float mean = warp_sum(s) * (1.0f / C);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float dx = v[i].x - mean, dy = v[i].y - mean, dz = v[i].z - mean, dw = v[i].w - mean;
    q += (dx * dx + dy * dy) + (dz * dz + dw * dw);
  }
  const float var = warp_sum(q) * (1.0f / C);
  const float rstd = rsqrtf(var + 1e-5f);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int c4 = lane + 32 * i;
    const float4 ww = __ldg(w4 + c4), bb = __ldg(b4 + c4);
    const float y0 = (v[i].x - mean) * rstd * ww.x + bb.x;
    const float y1 = (v[i].y - mean) * rstd * ww.y + bb.y;
    const float y2 = (v[i].z - mean) * rstd * ww.z + bb.z;
    const float y3 = (v[i].w - mean) * rstd * ww.w + bb.w;
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4*>(out + static_cast<size_t>(row) * C)[c4] = make_float4(y0, y1, y2, y3);
    } else {
      uint2 p;
      p.x = pack2<OutT>(y0, y1);
      p.y = pack2<OutT>(y2, y3);
      reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * C)[c4] = p;
    }
  }
  if (lane == 0) {
    if (mean_out) mean_out[row] = mean;
    if (rstd_out) rstd_out[row] = rstd;
  }
}

// Any C with C % 4 == 0: one block per row, three passes over the row
// (sum, centred sum of squares, output); the re-reads hit L1/L2.
template <typename OutT>
__global__ void __launch_bounds__(256) layernorm_block_kernel(OutT* __restrict__ out, float* __restrict__ mean_out,
                                                              float* __restrict__ rstd_out,
                                                              const float* __restrict__ inp,
                                                              const float* __restrict__ w,
                                                              const float* __restrict__ b, int C) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const float* x = inp + static_cast<size_t>(row) * C;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  auto block_sum = [&](float v) {
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = (lane < nw) ? red[lane] : 0.f;
    return warp_sum(t);
  };
  float s = 0.f;
  for (int c = threadIdx.x; c < C; c += blockDim.x) s += x[c];
  const float mean = block_sum(s) / C;
  float q = 0.f;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const float d = x[c] - mean;
    q += d * d;
  }
  const float rstd = rsqrtf(block_sum(q) / C + 1e-5f);
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const float y = (x[c] - mean) * rstd * w[c] + b[c];
    out[static_cast<size_t>(row) * C + c] = from_f32<OutT>(y);
  }
  if (threadIdx.x == 0) {
    if (mean_out) mean_out[row] = mean;
    if (rstd_out) rstd_out[row] = rstd;
  }
}

template <typename OutT>
static void layernorm_dispatch(OutT* out, float* mean, float* rstd, const float* inp, const float* w, const float* b,
                               int N, int C, cudaStream_t s) {
  const int rows_per_block = 8;
  const unsigned grid = static_cast<unsigned>((N + rows_per_block - 1) / rows_per_block);
  switch (C) {
    case 256: launch_pdl(layernorm_warp_kernel<2, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    case 512: launch_pdl(layernorm_warp_kernel<4, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    case 768: launch_pdl(layernorm_warp_kernel<6, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    case 1024: launch_pdl(layernorm_warp_kernel<8, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    case 1280: launch_pdl(layernorm_warp_kernel<10, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    case 1536: launch_pdl(layernorm_warp_kernel<12, OutT>, dim3(grid), dim3(256), 0, s, out, mean, rstd, inp, w, b, N); return;
    default: layernorm_block_kernel<OutT><<<N, 256, 0, s>>>(out, mean, rstd, inp, w, b, C); return;
  }
}

void launch_layernorm_f32(float* out, float* mean, float* rstd, const float* inp, const float* w, const float* b,
                          int N, int C, cudaStream_t s) {
  layernorm_dispatch<float>(out, mean, rstd, inp, w, b, N, C, s);
}

template <typename T>
void launch_layernorm_16(T* out, const float* inp, const float* w, const float* b, int N, int C, cudaStream_t s) {
  layernorm_dispatch<T>(out, nullptr, nullptr, inp, w, b, N, C, s);
}
template void launch_layernorm_16<__nv_bfloat16>(__nv_bfloat16*, const float*, const float*, const float*, int, int,
                                                 cudaStream_t);
template void launch_layernorm_16<__half>(__half*, const float*, const float*, const float*, int, int, cudaStream_t);

// grid of a grid-stride elementwise kernel: enough blocks for n work items,
// at most 8 per SM
static unsigned stream_grid(long long n4, int threads) {
  int sms = num_sms();
  long long want = (n4 + threads - 1) / threads;
  long long cap = static_cast<long long>(sms) * 8;
  return static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
}

// ------------------------------------------------ residual + LayerNorm
// x += y (the sublayer output, 16-bit) and out = LN(x) (16-bit) in one pass:
// the residual add of the attention and MLP projections, fused into the
// LayerNorm that reads x next.  One warp per row of C = 128 * kVec; x is
// written back unless write_x is false (the last LayerNorm).
template <int kVec, typename T16>
__global__ void __launch_bounds__(256) residual_layernorm_kernel(float* __restrict__ x, const T16* __restrict__ y,
                                                                 T16* __restrict__ out, const float* __restrict__ w,
                                                                 const float* __restrict__ b, int N, int write_x) {
  pdl_wait();
  pdl_trigger();
  constexpr int C = 128 * kVec;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= N) return;
  float4* x4 = reinterpret_cast<float4*>(x + static_cast<size_t>(row) * C);
  const uint2* y4 = reinterpret_cast<const uint2*>(y + static_cast<size_t>(row) * C);
  float4 v[kVec];
  uint2 yy[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    v[i] = x4[lane + 32 * i];
    yy[i] = __ldcs(y4 + lane + 32 * i);
  }
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const T16* h = reinterpret_cast<const T16*>(&yy[i]);
    v[i].x += to_f32(h[0]);
    v[i].y += to_f32(h[1]);
    v[i].z += to_f32(h[2]);
    v[i].w += to_f32(h[3]);
    if (write_x) x4[lane + 32 * i] = v[i];
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  const float mean = warp_sum(s) * (1.0f / C);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float dx = v[i].x - mean, dy = v[i].y - mean, dz = v[i].z - mean, dw = v[i].w - mean;
    q += (dx * dx + dy * dy) + (dz * dz + dw * dw);
  }
  const float rstd = rsqrtf(warp_sum(q) * (1.0f / C) + 1e-5f);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int c4 = lane + 32 * i;
    const float4 ww = __ldg(w4 + c4), bb = __ldg(b4 + c4);
    uint2 p;
    p.x = pack2<T16>((v[i].x - mean) * rstd * ww.x + bb.x, (v[i].y - mean) * rstd * ww.y + bb.y);
    p.y = pack2<T16>((v[i].z - mean) * rstd * ww.z + bb.z, (v[i].w - mean) * rstd * ww.w + bb.w);
    reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * C)[c4] = p;
  }
}

// x += y for any C (the fallback before a plain LayerNorm)
template <typename T16>
__global__ void add16_kernel(float* __restrict__ x, const T16* __restrict__ y, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    x[i] += to_f32(y[i]);
}

template <typename T16>
void launch_residual_layernorm_16(float* x, const T16* y, T16* out, const float* w, const float* b, int N, int C,
                                  bool write_x, cudaStream_t s) {
  const int rows_per_block = 8;
  const unsigned grid = static_cast<unsigned>((N + rows_per_block - 1) / rows_per_block);
  const int wx = write_x ? 1 : 0;
  switch (C) {
    case 256: launch_pdl(residual_layernorm_kernel<2, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    case 512: launch_pdl(residual_layernorm_kernel<4, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    case 768: launch_pdl(residual_layernorm_kernel<6, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    case 1024: launch_pdl(residual_layernorm_kernel<8, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    case 1280: launch_pdl(residual_layernorm_kernel<10, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    case 1536: launch_pdl(residual_layernorm_kernel<12, T16>, dim3(grid), dim3(256), 0, s, x, y, out, w, b, N, wx); return;
    default: {
      const long long n = static_cast<long long>(N) * C;
      add16_kernel<T16><<<stream_grid(n, 256), 256, 0, s>>>(x, y, n);
      launch_layernorm_16(out, x, w, b, N, C, s);
      return;
    }
  }
}
template void launch_residual_layernorm_16<__nv_bfloat16>(float*, const __nv_bfloat16*, __nv_bfloat16*,
                                                          const float*, const float*, int, int, bool, cudaStream_t);
template void launch_residual_layernorm_16<__half>(float*, const __half*, __half*, const float*, const float*, int,
                                                   int, bool, cudaStream_t);

// ------------------------------------------------------- GELU and residual
__global__ void gelu_kernel(float4* __restrict__ out, const float4* __restrict__ inp, long long n4) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = inp[i];
    out[i] = make_float4(gelu_exact(x.x), gelu_exact(x.y), gelu_exact(x.z), gelu_exact(x.w));
  }
}

__global__ void gelu_tail_kernel(float* __restrict__ out, const float* __restrict__ inp, int start, int n) {
  const int i = start + blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = gelu_exact(inp[i]);
}

__global__ void residual_kernel(float4* out, const float4* a, const float4* b, long long n4) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = a[i], y = b[i];
    out[i] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
  }
}

__global__ void residual_tail_kernel(float* out, const float* a, const float* b, int start, int n) {
  const int i = start + blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = a[i] + b[i];
}

void launch_gelu(float* out, const float* inp, int n, cudaStream_t s) {
  const long long n4 = n / 4;
  if (n4 > 0) gelu_kernel<<<stream_grid(n4, 256), 256, 0, s>>>(reinterpret_cast<float4*>(out),
                                                                reinterpret_cast<const float4*>(inp), n4);
  const int rem = n - static_cast<int>(n4 * 4);
  if (rem > 0) gelu_tail_kernel<<<1, 32, 0, s>>>(out, inp, static_cast<int>(n4 * 4), n);
}

void launch_residual(float* out, const float* a, const float* b, int n, cudaStream_t s) {
  const long long n4 = n / 4;
  if (n4 > 0)
    residual_kernel<<<stream_grid(n4, 256), 256, 0, s>>>(reinterpret_cast<float4*>(out),
                                                          reinterpret_cast<const float4*>(a),
                                                          reinterpret_cast<const float4*>(b), n4);
  const int rem = n - static_cast<int>(n4 * 4);
  if (rem > 0) residual_tail_kernel<<<1, 32, 0, s>>>(out, a, b, static_cast<int>(n4 * 4), n);
}

// ---------------------------------------------------------------- softmax
constexpr int kSoftmaxThreads = 1024;

// Combines two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void merge_stats(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;  // both empty
  s = s * __expf(m - mm) + s2 * __expf(m2 - mm);
  m = mm;
}

// Block-wide reduction of (max, sum) pairs; every thread gets the result.
__device__ __forceinline__ float2 block_merge_stats(float m, float s) {
  __shared__ float red_m[32], red_s[32];
  __shared__ float2 result;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    merge_stats(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  if (lane == 0) {
    red_m[wid] = m;
    red_s[wid] = s;
  }
  __syncthreads();
  if (wid == 0) {
    m = lane < nw ? red_m[lane] : -INFINITY;
    s = lane < nw ? red_s[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge_stats(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) result = make_float2(m, s);
  }
  __syncthreads();
  return result;
}

// Writes probs for one row given its max and 1/sum, streaming: four
// columns per thread and step, as a float4 (P = float) or as four 16-bit
// values (P = __half or __nv_bfloat16: each the fp32 probability rounded to
// nearest once, so they equal the fp32 output's values rounded).
template <typename P>
__device__ __forceinline__ void softmax_write_row(P* __restrict__ prow, const float4* __restrict__ lrow, int V,
                                                  int c4_lo, int c4_hi, float mx, float inv) {
  for (int c4 = c4_lo + static_cast<int>(threadIdx.x); c4 < c4_hi; c4 += blockDim.x) {
    const float4 x = __ldcs(lrow + c4);
    const int c = c4 * 4;
    float4 p;
    p.x = (c + 0 < V) ? __expf(x.x - mx) * inv : 0.f;
    p.y = (c + 1 < V) ? __expf(x.y - mx) * inv : 0.f;
    p.z = (c + 2 < V) ? __expf(x.z - mx) * inv : 0.f;
    p.w = (c + 3 < V) ? __expf(x.w - mx) * inv : 0.f;
    if constexpr (std::is_same<P, float>::value) {
      __stcs(reinterpret_cast<float4*>(prow) + c4, p);
    } else {
      __stcs(reinterpret_cast<uint2*>(prow) + c4, make_uint2(pack2<P>(p.x, p.y), pack2<P>(p.z, p.w)));
    }
  }
}

// Standalone softmax, one block per row: an online (max, sum) pass over the
// row, then the normalised write pass.  The second pass re-reads a row the
// block has just read; the rows in flight (a few MB) stay in L2, so HBM sees
// about one read and one write per element.
template <typename P>
__global__ void __launch_bounds__(kSoftmaxThreads) softmax_2pass_kernel(P* __restrict__ probs,
                                                                        const float4* __restrict__ logits, int V,
                                                                        int Vp4) {
  const size_t row = blockIdx.x;
  const float4* lrow = logits + row * Vp4;
  float m = -INFINITY, s = 0.f;
  for (int c4 = threadIdx.x; c4 < Vp4; c4 += blockDim.x) {
    const float4 x = lrow[c4];
    const int c = c4 * 4;
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (c + k >= V) continue;
      if (xs[k] > m) {
        s = s * __expf(m - xs[k]) + 1.f;
        m = xs[k];
      } else {
        s += __expf(xs[k] - m);
      }
    }
  }
  const float2 r = block_merge_stats(m, s);
  softmax_write_row(probs + row * Vp4 * 4, lrow, V, 0, Vp4, r.x, 1.0f / r.y);
}

void launch_softmax(void* probs, int probs_type, const float* logits, int N, int V, int Vp, cudaStream_t s) {
  const float4* l4 = reinterpret_cast<const float4*>(logits);
  switch (probs_type) {
    case kProbsF16:
      softmax_2pass_kernel<<<N, kSoftmaxThreads, 0, s>>>(static_cast<__half*>(probs), l4, V, Vp / 4);
      break;
    case kProbsBF16:
      softmax_2pass_kernel<<<N, kSoftmaxThreads, 0, s>>>(static_cast<__nv_bfloat16*>(probs), l4, V, Vp / 4);
      break;
    default:
      softmax_2pass_kernel<<<N, kSoftmaxThreads, 0, s>>>(static_cast<float*>(probs), l4, V, Vp / 4);
  }
}

// Softmax after the LM-head GEMM: the row's (max, sum) come from the
// per-tile statistics the GEMM epilogue left, so the logits are read once.
constexpr int kStatsThreads = 256;
template <typename P>
__global__ void __launch_bounds__(kStatsThreads) softmax_from_stats_kernel(P* __restrict__ probs,
                                                                           const float4* __restrict__ logits,
                                                                           const float2* __restrict__ stats,
                                                                           int tiles, int V, int Vp4) {
  pdl_wait();
  pdl_trigger();
  const size_t row = blockIdx.x;
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < tiles; i += blockDim.x) {
    const float2 p = stats[row * tiles + i];
    merge_stats(m, s, p.x, p.y);
  }
  const float2 r = block_merge_stats(m, s);
  // blockIdx.y: this block's share of the row's columns (one share unless
  // there are too few rows to fill the GPU)
  const int per = (Vp4 + static_cast<int>(gridDim.y) - 1) / static_cast<int>(gridDim.y);
  const int lo = static_cast<int>(blockIdx.y) * per;
  softmax_write_row(probs + row * Vp4 * 4, logits + row * Vp4, V, lo, min(Vp4, lo + per), r.x, 1.0f / r.y);
}

void launch_softmax_from_stats(void* probs, int probs_type, const float* logits, const float2* row_stats, int tiles,
                               int N, int V, int Vp, cudaStream_t s) {
  // a few rows (a decode step): split each row over blocks, about four
  // blocks per SM in all
  int split = N >= 4 * num_sms() ? 1 : (4 * num_sms() + N - 1) / N;
  if (split > 64) split = 64;
  const float4* l4 = reinterpret_cast<const float4*>(logits);
  const dim3 grid(N, split), block(kStatsThreads);
  switch (probs_type) {
    case kProbsF16:
      launch_pdl(softmax_from_stats_kernel<__half>, grid, block, 0, s, static_cast<__half*>(probs), l4, row_stats,
                 tiles, V, Vp / 4);
      break;
    case kProbsBF16:
      launch_pdl(softmax_from_stats_kernel<__nv_bfloat16>, grid, block, 0, s, static_cast<__nv_bfloat16*>(probs), l4,
                 row_stats, tiles, V, Vp / 4);
      break;
    default:
      launch_pdl(softmax_from_stats_kernel<float>, grid, block, 0, s, static_cast<float*>(probs), l4, row_stats,
                 tiles, V, Vp / 4);
  }
}

// ----------------------------------------------------------------- argmax
// One block per row; ties go to the smallest index.
__global__ void __launch_bounds__(512) argmax_kernel(int* __restrict__ next, const float* __restrict__ logits, int V,
                                                     int Vp) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sv[32];
  __shared__ int si[32];
  const float* row = logits + static_cast<size_t>(blockIdx.x) * Vp;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  auto take = [&](float x, int c) {
    if (x > best) {  // strictly greater: within a thread indices increase
      best = x;
      bi = c;
    }
  };
  int c0 = 0;  // columns below c0 are done by the vector loop
  if ((Vp & 3) == 0) {
    // 16-byte loads, four per thread per round so that they are in flight
    // together; a thread still visits its columns in increasing order
    const float4* row4 = reinterpret_cast<const float4*>(row);
    const int n4 = V / 4, stride = blockDim.x;
    for (int base = threadIdx.x; base < n4; base += 4 * stride) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (base + u * stride < n4) v[u] = __ldcs(row4 + base + u * stride);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (base + u * stride < n4) {
          const int c = 4 * (base + u * stride);
          take(v[u].x, c);
          take(v[u].y, c + 1);
          take(v[u].z, c + 2);
          take(v[u].w, c + 3);
        }
    }
    c0 = 4 * n4;
  }
  for (int c = c0 + threadIdx.x; c < V; c += blockDim.x) take(row[c], c);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (b2 > best || (b2 == best && i2 < bi)) {
      best = b2;
      bi = i2;
    }
  }
  if (lane == 0) {
    sv[wid] = best;
    si[wid] = bi;
  }
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (b2 > best || (b2 == best && i2 < bi)) {
        best = b2;
        bi = i2;
      }
    }
    if (lane == 0) next[blockIdx.x] = (bi == 0x7fffffff) ? 0 : bi;
  }
}

void launch_argmax(int* next, const float* logits, int B, int V, int Vp, cudaStream_t s) {
  launch_pdl(argmax_kernel, dim3(B), dim3(512), 0, s, next, logits, V, Vp);
}

// ------------------------------------------------------------ conversions
template <typename T>
__global__ void f32_to_16_kernel(T* __restrict__ out, const float* __restrict__ in, long long n) {
  const long long n4 = n / 4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = reinterpret_cast<const float4*>(in)[i];
    uint2 p;
    p.x = pack2<T>(x.x, x.y);
    p.y = pack2<T>(x.z, x.w);
    reinterpret_cast<uint2*>(out)[i] = p;
  }
  const long long i = n4 * 4 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (blockIdx.x == 0 && i < n) out[i] = from_f32<T>(in[i]);
}

template <typename T>
void launch_f32_to_16(T* out, const float* in, long long n, cudaStream_t s) {
  f32_to_16_kernel<T><<<stream_grid(n / 4 + 1, 256), 256, 0, s>>>(out, in, n);
}
template void launch_f32_to_16<__nv_bfloat16>(__nv_bfloat16*, const float*, long long, cudaStream_t);
template void launch_f32_to_16<__half>(__half*, const float*, long long, cudaStream_t);

// ----------------------------------------------------------- KV cache
// Copies keys and values of rows [0, T) of each sequence from the QKV buffer
// ([B*T, 3C], element type E) into a layer's cache halves at positions
// [0, T), through the cache's row layout (dense or paged).  One thread per
// 16 bytes of a head row.
template <typename E>
__global__ void kv_store_kernel(E* __restrict__ kc, E* __restrict__ vc, const E* __restrict__ qkv, int B, int T,
                                int C, int NH, KVRows rows) {
  pdl_wait();  // the QKV projection ahead has finished
  pdl_trigger();
  constexpr int kPer = 16 / sizeof(E);
  const int hs = C / NH;
  const int chunks = hs / kPer;
  const long long total = 2LL * B * T * NH * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    long long r = i;
    const int ch = static_cast<int>(r % chunks); r /= chunks;
    const int h = static_cast<int>(r % NH); r /= NH;
    const int t = static_cast<int>(r % T); r /= T;
    const int b = static_cast<int>(r % B); r /= B;
    const int kv = static_cast<int>(r);  // 0 = keys, 1 = values
    size_t row;
    if (rows.table == nullptr) {
      row = (static_cast<size_t>(b) * NH + h) * rows.maxT + t;
    } else {
      int blk = __ldg(rows.table + static_cast<size_t>(b) * rows.max_blocks + (t >> rows.lbs));
      if (blk < 0 || blk >= rows.num_blocks) {
        if (ch == 0 && h == 0) set_error(GPT2_DEVERR_BLOCK);
        continue;
      }
      row = ((static_cast<size_t>(blk) * NH + h) << rows.lbs) + (t & ((1 << rows.lbs) - 1));
    }
    const E* src = qkv + (static_cast<size_t>(b) * T + t) * 3 * C + (kv + 1) * C + h * hs + ch * kPer;
    E* dst = (kv == 0 ? kc : vc) + row * hs + ch * kPer;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

void launch_kv_store_f32(float* kc, float* vc, const float* qkv, int B, int T, int C, int NH, const KVRows& rows,
                         cudaStream_t s) {
  const long long total = 2LL * B * T * C / 4;
  launch_pdl(kv_store_kernel<float>, dim3(stream_grid(total, 256)), dim3(256), 0, s, kc, vc, qkv, B, T, C, NH, rows);
}

void launch_kv_store_16(uint16_t* kc, uint16_t* vc, const uint16_t* qkv, int B, int T, int C, int NH,
                        const KVRows& rows, cudaStream_t s) {
  const long long total = 2LL * B * T * C / 8;
  launch_pdl(kv_store_kernel<uint16_t>, dim3(stream_grid(total, 256)), dim3(256), 0, s, kc, vc, qkv, B, T, C, NH,
             rows);
}

}  // namespace gpt2
