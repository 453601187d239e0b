// attention_tc.cu -- causal attention of the GPT-2 forward pass on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); the computation follows Algorithm 1: key/value tiles stream
// through shared memory and each query row keeps a running maximum and sum
// while its unnormalised output accumulates, so the T x T score matrix never
// exists.  Key tiles after the query tile are never visited; only the
// diagonal tile is masked.
//
// One CTA per (query tile of 128 rows, head, sequence), two CTAs per SM:
//   warp 0      TMA: Q once, K tiles (2-stage) and V tiles (1 stage) of
//               128 keys x 64 dimensions, straight from the fused QKV buffer
//               viewed as [B][T][3C] (rows past T are zero-filled);
//   warp 1      TMEM (256 columns: S 128 x 128 fp32, O 128 x 64 fp32) and,
//               from one lane, S = Q K^T (4 x 128x128x16) and O += P V
//               (8 x 128x64x16, V as an MN-major operand);
//   warps 2-5   softmax, one thread per query row: read S from TMEM, mask,
//               running max, p = exp2(s - m) rounded to the 16-bit type into
//               swizzled shared memory (the A operand of P V), running sum;
//               O in TMEM is rescaled only when a row's maximum grows by
//               more than 2^8 (the stale maximum is exact as long as the
//               final division uses the same one); at the end O / l is
//               written to [B, T, C].
// Every wait is bounded; a timeout sets the device error word and the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kTQ = 128;  // query rows per CTA = TMEM lanes
constexpr int kTK = 128;  // keys per tile
constexpr int kHS = 64;   // head size
constexpr int kTileBytes = 128 * kHS * 2;  // 16 KB: 128 rows of 128 bytes
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;    // S: columns 0..127
constexpr uint32_t kTmemO = 128;  // O: columns 128..191
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Smem {
  static constexpr int q = 0;
  static constexpr int k = q + kTileBytes;       // 2 stages
  static constexpr int v = k + 2 * kTileBytes;   // 1 stage
  static constexpr int p = v + kTileBytes;       // keys 0-63, then keys 64-127
  static constexpr int bars = p + 2 * kTileBytes;
  // q_full, k_full[2], k_empty[2], v_full, v_empty, s_full, p_full, o_done, drain
  static constexpr int n_bars = 11;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(2 * (Smem::alloc + 1024) <= 233472, "two CTAs per SM");

template <typename T16, typename OutT>
__global__ void __launch_bounds__(kThreads, 2)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_qkv, OutT* __restrict__ out, int T, int C,
                     float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 6;
  uint64_t* s_full = bars + 7;
  uint64_t* p_full = bars + 8;
  uint64_t* o_done = bars + 9;
  uint64_t* drain = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = gridDim.x - 1 - blockIdx.x;  // longest query tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int n_kv = qt + 1;  // key tiles 0..qt (kTK == kTQ)
  constexpr uint32_t kFmt = std::is_same<T16, __half>::value ? 0u : 1u;
  constexpr uint32_t kIdescS = make_idesc(kFmt, kTQ, kTK);
  constexpr uint32_t kIdescPV = make_idesc(kFmt, kTQ, kHS) | (1u << 16);  // B (V) MN-major

  if (threadIdx.x == 0) {
    for (int i = 0; i < Smem::n_bars; ++i) mbar_init(&bars[i], i == 8 ? 4u : 1u);  // p_full: 4 softmax warps
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmap_qkv);
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      uint32_t k_filled = 0, k_par = 0;  // per stage: ever filled, parity of the last fill
      bool v_filled = false;
      uint32_t v_par = 0;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_3d(smem + Smem::q, &tmap_qkv, q_full, h * kHS, qt * kTQ, b);
      for (int j = 0; j < n_kv && !*abort_flag; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&k_empty[s], ((j >> 1) & 1) ^ 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], kTileBytes);
        tma_load_3d(smem + Smem::k + s * kTileBytes, &tmap_qkv, &k_full[s], C + h * kHS, j * kTK, b);
        k_filled |= 1u << s;
        k_par = (k_par & ~(1u << s)) | ((static_cast<uint32_t>(j >> 1) & 1u) << s);
        if (!mbar_wait(v_empty, (j & 1) ^ 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(v_full, kTileBytes);
        tma_load_3d(smem + Smem::v, &tmap_qkv, v_full, 2 * C + h * kHS, j * kTK, b);
        v_filled = true;
        v_par = j & 1;
      }
      // the copies issued here must land before the CTA can exit
      mbar_wait(q_full, 0);
      for (int s = 0; s < 2; ++s)
        if ((k_filled >> s) & 1u) mbar_wait(&k_full[s], (k_par >> s) & 1u);
      if (v_filled) mbar_wait(v_full, v_par);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0);
      const uint32_t q_addr = smem_u32(smem + Smem::q);
      const uint32_t p_addr = smem_u32(smem + Smem::p);
      const uint32_t v_addr = smem_u32(smem + Smem::v);
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j & 1;
        if (!(ok = mbar_wait(&k_full[s], (j >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + Smem::k + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHS / 16; ++kk)
          tc_mma<false>(tmem + kTmemS, smem_desc_sw128(q_addr + kk * 32), smem_desc_sw128(k_addr + kk * 32),
                        kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(&k_empty[s]);
        tc_commit(s_full);
        if (!(ok = mbar_wait(p_full, j & 1))) break;
        if (!(ok = mbar_wait(v_full, j & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          const uint32_t a = p_addr + (kk >> 2) * kTileBytes + (kk & 3) * 32;  // K-major P, 64-key atoms
          const uint32_t bv = v_addr + kk * 2048;                              // 16 keys = 2 groups of 8 rows
          tc_mma<false>(tmem + kTmemO, smem_desc_sw128(a), smem_desc_sw128_mn(bv, 1024), kIdescPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(v_empty);
        tc_commit(o_done);
      }
      if (!ok) *abort_flag = 1;
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within the tile = TMEM lane
    const int t = qt * kTQ + row;      // its position in the sequence
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    uint8_t* p0 = smem + Smem::p;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1)))) break;
      tc_fence_after();
      const bool diag = (j == n_kv - 1);
      const int key0 = j * kTK;
      // this row's keys in the tile: all 128, or on the diagonal tile those
      // at positions <= t and < T
      const int valid = diag ? max(0, min(min(t + 1, T) - key0, kTK)) : kTK;
      // the whole S row into registers: four loads, one wait
      uint32_t r[kTK];
#pragma unroll
      for (int c = 0; c < kTK / 32; ++c)
        tmem_ld_32x32b_x32(lane_base + kTmemS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
      tmem_ld_wait();
      float mx = -INFINITY;
      if (valid == kTK) {
#pragma unroll
        for (int e = 0; e < kTK; ++e) mx = fmaxf(mx, __uint_as_float(r[e]));
      } else {
#pragma unroll
        for (int e = 0; e < kTK; ++e)
          if (e < valid) mx = fmaxf(mx, __uint_as_float(r[e]));
      }
      const float m_new = fmaxf(m_run, mx * scale_log2);  // the scale is positive: it commutes with max
      // P and O are free once the previous P V has completed
      if (j > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1)))) break;
      const bool grow = (m_new - m_run) > kRescaleThreshold;  // true on the first tile
      if (__any_sync(0xffffffffu, grow)) {
        if (j > 0) {  // O holds P V of earlier tiles: scale it to the new maximum
          const float alpha = ex2(m_run - m_new);
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHS / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(lane_base + kTmemO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x32(lane_base + kTmemO + c * 32, o);
          }
          tmem_st_wait();
          l_run *= alpha;
        }
        m_run = m_new;
      }
      // p = exp2(s * scale - m), rounded to the 16-bit type, into P
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kTK / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int k = c * 32 + e;
          float p0v = ex2(fmaf(__uint_as_float(r[k]), scale_log2, -m_run));
          float p1v = ex2(fmaf(__uint_as_float(r[k + 1]), scale_log2, -m_run));
          if (valid != kTK) {
            if (k >= valid) p0v = 0.f;
            if (k + 1 >= valid) p1v = 0.f;
          }
          sum += p0v + p1v;
          pk[e >> 1] = pack2<T16>(p0v, p1v);
        }
        // 32 keys = 4 chunks of 16 bytes: atom c / 2, chunks (c % 2) * 4 + 0..3
        uint8_t* prow = p0 + (c >> 1) * kTileBytes + row * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (c & 1) * 4 + q;
          *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      l_run += sum;
      fence_proxy_async_smem();  // P written by this thread becomes visible to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_kv - 1) & 1));
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l_run;
      uint32_t o[64];
      {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_base + kTmemO, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = r[e];
        tmem_ld_32x32b_x32(lane_base + kTmemO + 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[32 + e] = r[e];
      }
      if (t < T) {
        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(b) * T + t) * C + h * kHS);
        if constexpr (std::is_same<OutT, float>::value) {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            dst[q] = make_uint4(__float_as_uint(__uint_as_float(o[4 * q + 0]) * inv),
                                __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv),
                                __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv),
                                __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv));
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint4 v;
            v.x = pack2<T16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            v.y = pack2<T16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            v.z = pack2<T16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            v.w = pack2<T16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            dst[q] = v;
          }
        }
      }
    } else {
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {
template <typename T16, typename OutT>
int launch_tc05_typed(void* out, const CUtensorMap& map, int B, int T, int C, int NH, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};  // per template instance and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_tc05_kernel<T16, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem::alloc) != cudaSuccess)
      return GPT2_ERR_CUDA;
    attr_set[dev] = true;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  dim3 grid((T + kTQ - 1) / kTQ, NH, B);
  attn_tc05_kernel<T16, OutT><<<grid, kThreads, Smem::alloc, s>>>(map, static_cast<OutT*>(out), T, C, scale_log2);
  return cudaPeekAtLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}
}  // namespace

// qkv [B,T,3C] of the 16-bit operand type op; out [B,T,C] of that type
// (out16) or fp32.  Head size 64 only.
int launch_attention_tc05(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                          cudaStream_t s) {
  if (C / NH != kHS || C % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  CUtensorMap map;
  const uint64_t dims[3] = {static_cast<uint64_t>(3 * C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[2] = {static_cast<uint64_t>(3 * C) * 2, static_cast<uint64_t>(T) * 3 * C * 2};
  const uint32_t box[3] = {kHS, kTK, 1};
  const CUtensorMapDataType dt = op == kOpF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tensor_map_sw128(&map, dt, 3, qkv, dims, strides, box)) return GPT2_ERR_CUDA;
  if (op == kOpF16)
    return out16 ? launch_tc05_typed<__half, __half>(out, map, B, T, C, NH, s)
                 : launch_tc05_typed<__half, float>(out, map, B, T, C, NH, s);
  return out16 ? launch_tc05_typed<__nv_bfloat16, __nv_bfloat16>(out, map, B, T, C, NH, s)
               : launch_tc05_typed<__nv_bfloat16, float>(out, map, B, T, C, NH, s);
}

}  // namespace gpt2
