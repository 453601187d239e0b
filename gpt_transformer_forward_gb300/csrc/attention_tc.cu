// attention_tc.cu -- causal attention of the GPT-2 forward pass on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); the computation follows Algorithm 1: key/value tiles stream
// through shared memory and each query row keeps a running maximum and sum
// while its unnormalised output accumulates, so the T x T score matrix never
// exists.  Key tiles after a query tile are never visited; only the diagonal
// tile is masked.
//
// One CTA per (pair of query tiles of 128 rows, head, sequence), one CTA per
// SM.  The two query tiles A = 2i and B = 2i + 1 share every key/value tile
// (B needs one more, its diagonal) and take turns on the tensor cores: while
// the softmax warps of A turn S_A into P_A, the tensor cores compute S_B and
// P_B V, and the other way round, so the exponentials of one tile hide the
// hand-offs of the other.
//   warp 0      TMA: both Q tiles, then K and V tiles of 128 keys x 64
//               dimensions (three stages each) straight from the fused QKV
//               buffer viewed as [B][T][3C] (rows past T are zero-filled);
//   warp 1      TMEM (S_A, S_B: 128 x 128 fp32; O_A, O_B: 128 x 64 fp32)
//               and, from one lane, S = Q K^T (4 x 128x128x16) and O += P V
//               (8 x 128x64x16, V as an MN-major operand);
//   warps 2-5   softmax of A, warps 6-9 softmax of B, one thread per query
//               row: the S row from TMEM (read twice in halves of 64
//               columns: once for the row maximum, once for the
//               exponentials), mask (diagonal tile only), running max,
//               p = exp2(s*scale - m) rounded to the 16-bit type into
//               swizzled shared memory (the A operand of P V), running sum;
//               O is rescaled in TMEM only when a row maximum grows by more
//               than 2^8 (exact: the final division uses the same stale
//               maximum); at the end O / l goes to [B, T, C].
// Every wait is bounded; a timeout sets the device error word and the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kTQ = 128;   // query rows per query tile = TMEM lanes
constexpr int kTK = 128;   // keys per key tile
constexpr int kHS = 64;    // head size
constexpr int kTileBytes = 128 * kHS * 2;  // 16 KB: 128 rows of 128 bytes
constexpr int kKV = 3;     // K and V pipeline stages
constexpr int kThreads = 64 + 2 * 128;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of query tile x at 128 x, O of query tile x at 256 + 64 x
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Smem {
  static constexpr int q = 0;                        // 2 query tiles
  static constexpr int k = q + 2 * kTileBytes;       // kKV stages
  static constexpr int v = k + kKV * kTileBytes;     // kKV stages
  static constexpr int p = v + kKV * kTileBytes;     // per query tile: keys 0-63, keys 64-127
  static constexpr int bars = p + 4 * kTileBytes;
  // q_full; k_full[kKV], k_empty[kKV], v_full[kKV], v_empty[kKV]; per query
  // tile: s_full, p_full, o_done; drain
  static constexpr int n_bars = 1 + 4 * kKV + 3 * 2 + 1;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(Smem::alloc <= 232448, "shared memory budget");

// 320 threads = 10 warps, one CTA per SM.  Registers are allotted per SM
// sub-partition (16K each, warps placed round-robin), so the sub-partition
// holding three warps caps a thread at 168 registers; the softmax threads
// therefore read their S row in halves instead of holding all of it.
template <typename T16, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_qkv, OutT* __restrict__ out, int T, int C,
                     float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;              // [kKV]
  uint64_t* k_empty = k_full + kKV;         // [kKV]
  uint64_t* v_full = k_empty + kKV;         // [kKV]
  uint64_t* v_empty = v_full + kKV;         // [kKV]
  uint64_t* s_full = v_empty + kKV;         // [query tile]: S of its key tile j completes phase j
  uint64_t* p_full = s_full + 2;            // [query tile], one arrival per softmax warp
  uint64_t* o_done = p_full + 2;            // [query tile]: P V of key tile j completes phase j
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = gridDim.x - 1 - blockIdx.x;  // longest pairs first
  const int h = blockIdx.y, b = blockIdx.z;
  const int qt0 = 2 * pair;                     // query tile A; B = qt0 + 1
  const int n_a = qt0 + 1, n_b = qt0 + 2;       // key tiles of A and B (kTK == kTQ)
  constexpr uint32_t kFmt = std::is_same<T16, __half>::value ? 0u : 1u;
  constexpr uint32_t kIdescS = make_idesc(kFmt, kTQ, kTK);
  constexpr uint32_t kIdescPV = make_idesc(kFmt, kTQ, kHS) | (1u << 16);  // B (V) MN-major

  if (threadIdx.x == 0) {
    for (int i = 0; i < Smem::n_bars; ++i) mbar_init(&bars[i], 1u);
    mbar_init(&p_full[0], 4u);
    mbar_init(&p_full[1], 4u);
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
      uint32_t k_filled = 0, k_par = 0, v_filled = 0, v_par = 0;  // per stage: filled, parity of last fill
      mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
      tma_load_3d(smem + Smem::q, &tmap_qkv, q_full, h * kHS, qt0 * kTQ, b);
      tma_load_3d(smem + Smem::q + kTileBytes, &tmap_qkv, q_full, h * kHS, (qt0 + 1) * kTQ, b);
      for (int j = 0; j < n_b && !*abort_flag; ++j) {
        const int s = j % kKV;
        const uint32_t ph = (j / kKV) & 1;
        if (!mbar_wait(&k_empty[s], ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], kTileBytes);
        tma_load_3d(smem + Smem::k + s * kTileBytes, &tmap_qkv, &k_full[s], C + h * kHS, j * kTK, b);
        k_filled |= 1u << s;
        k_par = (k_par & ~(1u << s)) | (ph << s);
        if (!mbar_wait(&v_empty[s], ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&v_full[s], kTileBytes);
        tma_load_3d(smem + Smem::v + s * kTileBytes, &tmap_qkv, &v_full[s], 2 * C + h * kHS, j * kTK, b);
        v_filled |= 1u << s;
        v_par = (v_par & ~(1u << s)) | (ph << s);
      }
      // the copies issued here must land before the CTA can exit
      mbar_wait(q_full, 0);
      for (int s = 0; s < kKV; ++s) {
        if ((k_filled >> s) & 1u) mbar_wait(&k_full[s], (k_par >> s) & 1u);
        if ((v_filled >> s) & 1u) mbar_wait(&v_full[s], (v_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0);
      const uint32_t q_addr = smem_u32(smem + Smem::q);
      const uint32_t p_addr = smem_u32(smem + Smem::p);
      // S_x = Q_x K_j^T into TMEM S of query tile x
      auto issue_s = [&](int x, int j) {
        const uint32_t k_addr = smem_u32(smem + Smem::k + (j % kKV) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHS / 16; ++kk)
          tc_mma<false>(tmem + kTmemS + x * kTK, smem_desc_sw128(q_addr + x * kTileBytes + kk * 32),
                        smem_desc_sw128(k_addr + kk * 32), kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[x]);
      };
      // O_x += P_x V_j
      auto issue_pv = [&](int x, int j) {
        const uint32_t v_addr = smem_u32(smem + Smem::v + (j % kKV) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          const uint32_t a = p_addr + x * 2 * kTileBytes + (kk >> 2) * kTileBytes + (kk & 3) * 32;
          const uint32_t bv = v_addr + kk * 2048;  // 16 keys = 2 groups of 8 rows
          tc_mma<false>(tmem + kTmemO + x * kHS, smem_desc_sw128(a), smem_desc_sw128_mn(bv, 1024), kIdescPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&o_done[x]);
      };
      if (ok && (ok = mbar_wait(&k_full[0], 0))) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        tc_commit(&k_empty[0]);
      }
      for (int j = 0; j < n_b && ok; ++j) {
        if (!(ok = mbar_wait(&v_full[j % kKV], (j / kKV) & 1))) break;
        bool k_next = false;  // K_{j+1} already waited for
        if (j < n_a) {        // query tile A: P V of tile j, then S of tile j + 1
          if (!(ok = mbar_wait(&p_full[0], j & 1))) break;
          tc_fence_after();
          issue_pv(0, j);
          if (j + 1 < n_a) {
            if (!(ok = mbar_wait(&k_full[(j + 1) % kKV], ((j + 1) / kKV) & 1))) break;
            k_next = true;
            tc_fence_after();
            issue_s(0, j + 1);
          }
        }
        // query tile B: P V of tile j, then S of tile j + 1
        if (!(ok = mbar_wait(&p_full[1], j & 1))) break;
        tc_fence_after();
        issue_pv(1, j);
        tc_commit(&v_empty[j % kKV]);  // both query tiles have used V_j
        if (j + 1 < n_b) {
          if (!k_next && !(ok = mbar_wait(&k_full[(j + 1) % kKV], ((j + 1) / kKV) & 1))) break;
          tc_fence_after();
          issue_s(1, j + 1);
          tc_commit(&k_empty[(j + 1) % kKV]);  // both query tiles have used K_{j+1}
        }
      }
      if (!ok) *abort_flag = 1;
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int x = (warp - 2) >> 2;           // query tile: 0 = A (warps 2-5), 1 = B (warps 6-9)
    const int quad = warp & 3;               // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;        // query row within the tile = TMEM lane
    const int t = (qt0 + x) * kTQ + row;     // its position in the sequence
    const int n_x = x == 0 ? n_a : n_b;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t s_col = kTmemS + x * kTK;
    uint8_t* pbase = smem + Smem::p + x * 2 * kTileBytes + row * 128;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_x; ++j) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1)))) break;
      tc_fence_after();
      const int key0 = j * kTK;
      // this row's keys in the tile: all 128, or on the diagonal tile those
      // at positions <= t and < T
      const int valid = (j == n_x - 1) ? max(0, min(min(t + 1, T) - key0, kTK)) : kTK;
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // pass 1: the row maximum
        uint32_t r[64];
        tmem_ld_32x32b_x32(lane_base + s_col + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld_32x32b_x32(lane_base + s_col + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
        if (valid == kTK) {
#pragma unroll
          for (int e = 0; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(r[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (half * 64 + e < valid) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(r[e]));
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_run, mx * scale_log2);  // the scale is positive: it commutes with max
      // P V of tile j - 1 must be done: P is overwritten below and O may be rescaled
      if (j > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[x], (j - 1) & 1)))) break;
      const bool grow = (m_new - m_run) > kRescaleThreshold;  // true on the first tile
      if (__any_sync(0xffffffffu, grow)) {
        if (j > 0) {
          tc_fence_after();
          const float alpha = ex2(m_run - m_new);
#pragma unroll 1
          for (int c = 0; c < kHS / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(lane_base + kTmemO + x * kHS + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x32(lane_base + kTmemO + x * kHS + c * 32, o);
          }
          tmem_st_wait();
          l_run *= alpha;
        }
        m_run = m_new;
      }
      // pass 2: p = exp2(s * scale - m), rounded to the 16-bit type, into P_x
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r[64];
        tmem_ld_32x32b_x32(lane_base + s_col + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld_32x32b_x32(lane_base + s_col + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = half * 2 + c2;  // 32-key chunk of the tile
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int k = c * 32 + e;
            float p0v = ex2(fmaf(__uint_as_float(r[c2 * 32 + e]), scale_log2, -m_run));
            float p1v = ex2(fmaf(__uint_as_float(r[c2 * 32 + e + 1]), scale_log2, -m_run));
            if (valid != kTK) {
              if (k >= valid) p0v = 0.f;
              if (k + 1 >= valid) p1v = 0.f;
            }
            sum4[(e >> 1) & 3] += p0v + p1v;
            pk[e >> 1] = pack2<T16>(p0v, p1v);
          }
          // 32 keys = 4 chunks of 16 bytes: atom c / 2, chunks (c % 2) * 4 + 0..3
          uint8_t* prow = pbase + (c >> 1) * kTileBytes;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (c & 1) * 4 + q;
            *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      l_run += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      fence_proxy_async_smem();  // P written by this thread becomes visible to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[x], (n_x - 1) & 1));
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l_run;
#pragma unroll 1
      for (int c = 0; c < kHS / 32; ++c) {  // O / l, 32 columns at a time
        uint32_t o[32];
        tmem_ld_32x32b_x32(lane_base + kTmemO + x * kHS + c * 32, o);
        tmem_ld_wait();
        if (t < T) {
          OutT* dst = out + (static_cast<size_t>(b) * T + t) * C + h * kHS + c * 32;
          if constexpr (std::is_same<OutT, float>::value) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<uint4*>(dst)[q] =
                  make_uint4(__float_as_uint(__uint_as_float(o[4 * q + 0]) * inv),
                             __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv),
                             __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv),
                             __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv));
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack2<T16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
              v.y = pack2<T16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
              v.z = pack2<T16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
              v.w = pack2<T16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
              reinterpret_cast<uint4*>(dst)[q] = v;
            }
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
    const cudaError_t e = cudaFuncSetAttribute(attn_tc05_kernel<T16, OutT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  dim3 grid((T + 2 * kTQ - 1) / (2 * kTQ), NH, B);  // pairs of query tiles
  attn_tc05_kernel<T16, OutT><<<grid, kThreads, Smem::alloc, s>>>(map, static_cast<OutT*>(out), T, C, scale_log2);
  const cudaError_t e = cudaPeekAtLastError();
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
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
