// attention_bwd.cu -- the backward pass of causal multi-head attention, in
// fp32 on the CUDA cores ("Understand FlashAttention (II)": the backward
// algorithm of FlashAttention's Algorithm 1).
//
// With S = Q K^T * scale (causal), P = softmax_rows(S), O = P V and the
// incoming gradient dO, the gradients are
//   dV = P^T dO,  dP = dO V^T,  dS = P (dP - D),  dQ = dS K * scale,
//   dK = dS^T Q * scale,   D[t] = sum_d dO[t][d] O[t][d],
// and P is recomputed tile by tile from the row statistic L = max + log(sum)
// of the forward's softmax (P = exp(S - L)), so that no T x T matrix is
// stored.  Three kernels, each over 64-row tiles of one (sequence, head):
//   stats   per query tile: L of every row (an online maximum and sum over
//           its key tiles) and D;
//   dk_dv   per key tile: loops over the query tiles that see it,
//           accumulating dK and dV in registers;
//   dq      per query tile: loops over the key tiles it sees, accumulating
//           dQ in registers.
// Splitting dK/dV and dQ into two kernels recomputes S and dP once more but
// needs no atomics: every gradient element is written once, by one thread,
// so results are deterministic.  Tiles are staged in shared memory as fp32
// with rows padded to an odd number of words (conflict-free column reads);
// 256 threads each own a 4 x 4 block of a 64 x 64 score tile (rows
// ty + 16a, columns tx + 16b) and a 4 x hs/16 block of a gradient tile.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kBT = 64;            // rows of a tile
constexpr int kBwdThreads = 256;   // 16 x 16

template <int HS>
struct BwdTiles {
  static constexpr int kLd = HS + 1;                   // padded row of a head-dimension tile
  static constexpr int kTile = kBT * kLd;              // floats
  static constexpr int kSq = kBT * (kBT + 1);          // a padded 64 x 64 tile
};

// rows [r0, r0 + 64) of a [rows, stride] fp32 matrix, columns [0, HS) from
// src, into dst[64][HS + 1]; rows at or past T read as zero
template <int HS>
__device__ __forceinline__ void load_tile(float* dst, const float* __restrict__ src, size_t stride, int r0, int T) {
  for (int i = threadIdx.x; i < kBT * HS; i += kBwdThreads) {
    const int r = i / HS, d = i % HS;
    dst[r * BwdTiles<HS>::kLd + d] = (r0 + r < T) ? __ldg(src + static_cast<size_t>(r0 + r) * stride + d) : 0.f;
  }
}

// S[a][b] = sum_d X[ty + 16a][d] Y[tx + 16b][d] over two padded tiles
template <int HS>
__device__ __forceinline__ void tile_dot(float (&s)[4][4], const float* X, const float* Y, int ty, int tx) {
  constexpr int ld = BwdTiles<HS>::kLd;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) s[a][b] = 0.f;
#pragma unroll 8
  for (int d = 0; d < HS; ++d) {
    float xa[4], yb[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) xa[a] = X[(ty + 16 * a) * ld + d];
#pragma unroll
    for (int b = 0; b < 4; ++b) yb[b] = Y[(tx + 16 * b) * ld + d];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) s[a][b] = fmaf(xa[a], yb[b], s[a][b]);
  }
}

// The forward's row statistic L = m + log(l) of every query row of a tile,
// and D = sum_d dO O.  Grid (query tiles, NH, B).
template <int HS>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_stats_kernel(float* __restrict__ Lrow, float* __restrict__ Drow,
                                                                     const float* __restrict__ qkv,
                                                                     const float* __restrict__ out,
                                                                     const float* __restrict__ dout, int T, int C,
                                                                     float scale) {
  using Tl = BwdTiles<HS>;
  __shared__ float Qs[Tl::kTile], Ks[Tl::kTile];
  const int i0 = blockIdx.x * kBT, h = blockIdx.y, b = blockIdx.z, NH = gridDim.y;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* base = qkv + static_cast<size_t>(b) * T * 3 * C;
  load_tile<HS>(Qs, base + h * HS, 3 * C, i0, T);
  float m[4], l[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
  }
  const int j_end = min(i0 + kBT, T);  // keys < j_end can be visible to this tile
  for (int j0 = 0; j0 < j_end; j0 += kBT) {
    __syncthreads();
    load_tile<HS>(Ks, base + C + h * HS, 3 * C, j0, T);
    __syncthreads();
    float s[4][4];
    tile_dot<HS>(s, Qs, Ks, ty, tx);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int t = i0 + ty + 16 * a;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx + 16 * c;
        s[a][c] = (j <= t && j < T) ? s[a][c] * scale : -INFINITY;
        mx = fmaxf(mx, s[a][c]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));  // the row's 16 lanes
      const float m_new = fmaxf(m[a], mx);
      // (every lane of the warp reaches the shuffles; a row with no visible
      // key so far keeps m = -inf and l = 0)
      const float m_ref = m_new == -INFINITY ? 0.f : m_new;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) sum += expf(s[a][c] - m_ref);  // exp(-inf) = 0
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (m_new != -INFINITY) {
        l[a] = l[a] * expf(m[a] - m_new) + sum;
        m[a] = m_new;
      }
    }
  }
  const size_t row0 = (static_cast<size_t>(b) * NH + h) * T;
  if (tx == 0) {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int t = i0 + ty + 16 * a;
      if (t < T) Lrow[row0 + t] = m[a] + logf(l[a]);
    }
  }
  // D: four threads per row, a quarter of the head's dimensions each
  const int r = threadIdx.x >> 2, qd = threadIdx.x & 3;
  const int t = i0 + r;
  float dd = 0.f;
  if (t < T) {
    const float* go = dout + (static_cast<size_t>(b) * T + t) * C + h * HS;
    const float* o = out + (static_cast<size_t>(b) * T + t) * C + h * HS;
#pragma unroll
    for (int d = qd * (HS / 4); d < (qd + 1) * (HS / 4); ++d) dd = fmaf(__ldg(go + d), __ldg(o + d), dd);
  }
  dd += __shfl_xor_sync(0xffffffffu, dd, 1);
  dd += __shfl_xor_sync(0xffffffffu, dd, 2);
  if (qd == 0 && t < T) Drow[row0 + t] = dd;
}

// dK and dV of one key tile.  Grid (key tiles, NH, B); dynamic shared
// memory: K, V, Q, dO tiles, P^T and dS^T, L and D of the query tile.
template <int HS>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_dkdv_kernel(float* __restrict__ dqkv,
                                                                    const float* __restrict__ qkv,
                                                                    const float* __restrict__ dout,
                                                                    const float* __restrict__ Lrow,
                                                                    const float* __restrict__ Drow, int T, int C,
                                                                    float scale) {
  using Tl = BwdTiles<HS>;
  constexpr int ND = HS / 16;  // head dimensions per thread
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + Tl::kTile;
  float* Qs = Vs + Tl::kTile;
  float* Os = Qs + Tl::kTile;  // dO
  float* Ps = Os + Tl::kTile;  // P^T [key][query]
  float* Ss = Ps + Tl::kSq;    // dS^T [key][query]
  float* Ls = Ss + Tl::kSq;
  float* Ds = Ls + kBT;
  const int j0 = blockIdx.x * kBT, h = blockIdx.y, b = blockIdx.z, NH = gridDim.y;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* base = qkv + static_cast<size_t>(b) * T * 3 * C;
  const float* gbase = dout + static_cast<size_t>(b) * T * C;
  const size_t row0 = (static_cast<size_t>(b) * NH + h) * T;
  load_tile<HS>(Ks, base + C + h * HS, 3 * C, j0, T);
  load_tile<HS>(Vs, base + 2 * C + h * HS, 3 * C, j0, T);
  float dk[4][ND], dv[4][ND];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int e = 0; e < ND; ++e) dk[a][e] = dv[a][e] = 0.f;
  for (int i0 = j0; i0 < T; i0 += kBT) {  // the query tiles at or after the key tile see it
    __syncthreads();
    load_tile<HS>(Qs, base + h * HS, 3 * C, i0, T);
    load_tile<HS>(Os, gbase + h * HS, C, i0, T);
    if (threadIdx.x < kBT) {
      const int t = i0 + threadIdx.x;
      Ls[threadIdx.x] = t < T ? __ldg(Lrow + row0 + t) : 0.f;
      Ds[threadIdx.x] = t < T ? __ldg(Drow + row0 + t) : 0.f;
    }
    __syncthreads();
    // S^T and dP^T: rows = keys (ty + 16a), columns = queries (tx + 16c)
    float st[4][4], dpt[4][4];
    tile_dot<HS>(st, Ks, Qs, ty, tx);
    tile_dot<HS>(dpt, Vs, Os, ty, tx);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + ty + 16 * a, t = i0 + tx + 16 * c;
        const float p = (j <= t && t < T && j < T) ? expf(st[a][c] * scale - Ls[tx + 16 * c]) : 0.f;
        Ps[(ty + 16 * a) * (kBT + 1) + tx + 16 * c] = p;
        Ss[(ty + 16 * a) * (kBT + 1) + tx + 16 * c] = p * (dpt[a][c] - Ds[tx + 16 * c]);
      }
    __syncthreads();
    // dV += P^T dO, dK += dS^T Q: rows = keys (ty + 16a), columns = head
    // dimensions (tx + 16e)
#pragma unroll 4
    for (int r = 0; r < kBT; ++r) {
      float pa[4], sa[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        pa[a] = Ps[(ty + 16 * a) * (kBT + 1) + r];
        sa[a] = Ss[(ty + 16 * a) * (kBT + 1) + r];
      }
#pragma unroll
      for (int e = 0; e < ND; ++e) {
        const float o = Os[r * Tl::kLd + tx + 16 * e], q = Qs[r * Tl::kLd + tx + 16 * e];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          dv[a][e] = fmaf(pa[a], o, dv[a][e]);
          dk[a][e] = fmaf(sa[a], q, dk[a][e]);
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + ty + 16 * a;
    if (j >= T) continue;
    float* g = dqkv + (static_cast<size_t>(b) * T + j) * 3 * C + h * HS;
#pragma unroll
    for (int e = 0; e < ND; ++e) {
      g[C + tx + 16 * e] = dk[a][e] * scale;
      g[2 * C + tx + 16 * e] = dv[a][e];
    }
  }
}

// dQ of one query tile.  Grid (query tiles, NH, B); dynamic shared memory:
// Q, dO, K, V tiles, dS, L and D of the tile.
template <int HS>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_dq_kernel(float* __restrict__ dqkv,
                                                                  const float* __restrict__ qkv,
                                                                  const float* __restrict__ dout,
                                                                  const float* __restrict__ Lrow,
                                                                  const float* __restrict__ Drow, int T, int C,
                                                                  float scale) {
  using Tl = BwdTiles<HS>;
  constexpr int ND = HS / 16;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Os = Qs + Tl::kTile;  // dO
  float* Ks = Os + Tl::kTile;
  float* Vs = Ks + Tl::kTile;
  float* Ss = Vs + Tl::kTile;  // dS [query][key]
  float* Ls = Ss + Tl::kSq;
  float* Ds = Ls + kBT;
  const int i0 = blockIdx.x * kBT, h = blockIdx.y, b = blockIdx.z, NH = gridDim.y;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* base = qkv + static_cast<size_t>(b) * T * 3 * C;
  const size_t row0 = (static_cast<size_t>(b) * NH + h) * T;
  load_tile<HS>(Qs, base + h * HS, 3 * C, i0, T);
  load_tile<HS>(Os, dout + static_cast<size_t>(b) * T * C + h * HS, C, i0, T);
  if (threadIdx.x < kBT) {
    const int t = i0 + threadIdx.x;
    Ls[threadIdx.x] = t < T ? __ldg(Lrow + row0 + t) : 0.f;
    Ds[threadIdx.x] = t < T ? __ldg(Drow + row0 + t) : 0.f;
  }
  float dq[4][ND];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int e = 0; e < ND; ++e) dq[a][e] = 0.f;
  const int j_end = min(i0 + kBT, T);
  for (int j0 = 0; j0 < j_end; j0 += kBT) {
    __syncthreads();
    load_tile<HS>(Ks, base + C + h * HS, 3 * C, j0, T);
    load_tile<HS>(Vs, base + 2 * C + h * HS, 3 * C, j0, T);
    __syncthreads();
    // S and dP: rows = queries (ty + 16a), columns = keys (tx + 16c)
    float s[4][4], dp[4][4];
    tile_dot<HS>(s, Qs, Ks, ty, tx);
    tile_dot<HS>(dp, Os, Vs, ty, tx);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = i0 + ty + 16 * a, j = j0 + tx + 16 * c;
        const float p = (j <= t && t < T && j < T) ? expf(s[a][c] * scale - Ls[ty + 16 * a]) : 0.f;
        Ss[(ty + 16 * a) * (kBT + 1) + tx + 16 * c] = p * (dp[a][c] - Ds[ty + 16 * a]);
      }
    __syncthreads();
    // dQ += dS K: rows = queries (ty + 16a), columns = head dimensions
#pragma unroll 4
    for (int c = 0; c < kBT; ++c) {
      float sa[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sa[a] = Ss[(ty + 16 * a) * (kBT + 1) + c];
#pragma unroll
      for (int e = 0; e < ND; ++e) {
        const float k = Ks[c * Tl::kLd + tx + 16 * e];
#pragma unroll
        for (int a = 0; a < 4; ++a) dq[a][e] = fmaf(sa[a], k, dq[a][e]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int t = i0 + ty + 16 * a;
    if (t >= T) continue;
    float* g = dqkv + (static_cast<size_t>(b) * T + t) * 3 * C + h * HS;
#pragma unroll
    for (int e = 0; e < ND; ++e) g[tx + 16 * e] = dq[a][e] * scale;
  }
}

template <int HS>
int attention_backward_hs(float* dqkv, const float* dout, const float* qkv, const float* out, float* Lrow,
                          float* Drow, int B, int T, int C, int NH, cudaStream_t s) {
  using Tl = BwdTiles<HS>;
  constexpr size_t kSmemKV = (4 * Tl::kTile + 2 * Tl::kSq + 2 * kBT) * sizeof(float);
  constexpr size_t kSmemQ = (4 * Tl::kTile + Tl::kSq + 2 * kBT) * sizeof(float);
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<HS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemKV));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dq_kernel<HS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemQ));
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  const float scale = 1.0f / sqrtf(static_cast<float>(HS));
  const dim3 grid((T + kBT - 1) / kBT, NH, B);
  attn_bwd_stats_kernel<HS><<<grid, kBwdThreads, 0, s>>>(Lrow, Drow, qkv, out, dout, T, C, scale);
  attn_bwd_dkdv_kernel<HS><<<grid, kBwdThreads, kSmemKV, s>>>(dqkv, qkv, dout, Lrow, Drow, T, C, scale);
  attn_bwd_dq_kernel<HS><<<grid, kBwdThreads, kSmemQ, s>>>(dqkv, qkv, dout, Lrow, Drow, T, C, scale);
  return GPT2_OK;
}

}  // namespace

int launch_attention_backward(float* dqkv, const float* dout, const float* qkv, const float* out, float* Lrow,
                              float* Drow, int B, int T, int C, int NH, cudaStream_t s) {
  switch (C / NH) {
    case 16: return attention_backward_hs<16>(dqkv, dout, qkv, out, Lrow, Drow, B, T, C, NH, s);
    case 32: return attention_backward_hs<32>(dqkv, dout, qkv, out, Lrow, Drow, B, T, C, NH, s);
    case 64: return attention_backward_hs<64>(dqkv, dout, qkv, out, Lrow, Drow, B, T, C, NH, s);
  }
  return GPT2_ERR_UNSUPPORTED;
}

}  // namespace gpt2
