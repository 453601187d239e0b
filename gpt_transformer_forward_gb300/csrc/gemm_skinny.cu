// gemm_skinny.cu -- the GEMM sites at a few activation rows (M <= 64: the
// decode step's one token per sequence, small forward passes) on tcgen05.
//
//   D[M, N] = A[M, K] W[N, K]^T, computed as D^T = W A^T
//
// At M this small the weights are nearly all of the traffic, and the
// 128 x 256 tiles of the main GEMM kernel leave most SMs idle (N / 256 CTAs,
// each streaming a long K range).  Here the MMA's M side is 128 weight rows
// and its N side the M activation rows padded to a multiple of 16, and the K
// range of each 128-row weight block is split over the s CTAs of a
// thread-block cluster (s a power of two up to 16), so that about one CTA per
// SM streams its share of the weights.  Each CTA (128 threads):
//   warp 0  lane 0: TMA of 128 weight rows x 128 bytes of K and of the padded
//           activation rows x 128 bytes per stage (128-byte swizzle), a
//           four-stage ring;
//   warp 1  allocates 64 TMEM columns and issues the MMAs (128 x n x 16 for
//           16-bit operands, x 8 for tf32; one elected lane);
//   all     tcgen05.ld of the partial D^T (thread = weight row, registers =
//           activation rows) into shared memory as [m][128] fp32, over the
//           stage buffers, which the finished MMAs no longer read.
// After a cluster barrier, CTA r sums its 1/s slice of the block over the
// cluster's s partials (distributed shared memory, in rank order, so the
// result does not depend on timing), adds the bias, applies the epilogue and
// stores with plain vector stores; a second cluster barrier keeps every
// CTA's shared memory alive until its peers have read it.
// Launched as a programmatic dependent launch (in a decode step), a CTA
// sets up and requests its first weight tiles before it waits for the
// kernel ahead of it.
// Every mbarrier wait is bounded; on a timeout the CTA records
// GPT2_DEVERR_TIMEOUT and still reaches both cluster barriers.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kSkRowsW = 128;             // weight rows per block (the MMA's M)
constexpr int kSkMaxRows = 64;            // activation rows (the MMA's N, at most)
constexpr int kSkRowBytes = 128;          // K bytes per stage (one swizzle row)
constexpr int kSkStages = 4;
constexpr int kSkWStage = kSkRowsW * kSkRowBytes;    // 16 KB
constexpr int kSkXStage = kSkMaxRows * kSkRowBytes;  // 8 KB
constexpr int kSkThreads = 128;
constexpr int kSkTmemCols = 64;
constexpr int kSkMaxSplits = 16;
constexpr int kSkXOff = kSkStages * kSkWStage;
constexpr int kSkBarOff = kSkXOff + kSkStages * kSkXStage;
constexpr int kSkMiscOff = kSkBarOff + (2 * kSkStages + 1) * 8;
constexpr int kSkAlloc = kSkMiscOff + 16 + 1024;  // + slack for 1024-byte alignment
static_assert(kSkMaxRows * kSkRowsW * 4 <= kSkBarOff, "the partial fits over the stage buffers");

template <int kEpi, int kOp>
__global__ void __launch_bounds__(kSkThreads)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                       void* __restrict__ out, const float* __restrict__ bias, int M, int N, int K, int n_mma,
                       uint32_t idesc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSkBarOff);
  uint64_t* empty = full + kSkStages;
  uint64_t* done = empty + kSkStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSkMiscOff);

  constexpr bool kTF32 = (kOp == kOpTF32);
  constexpr int kElemBytes = kTF32 ? 4 : 2;
  constexpr int kBK = kSkRowBytes / kElemBytes;  // K elements per stage
  constexpr int kMmaK = 32 / kElemBytes;         // K per instruction (32 bytes)
  using Out16 = typename std::conditional<kOp == kOpF16, __half, __nv_bfloat16>::type;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the cluster is the s CTAs sharing one weight block; rank = K split
  uint32_t n_splits;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n_splits));
  const uint32_t rank = cluster_ctarank();
  const int n_blk = static_cast<int>(blockIdx.x) / static_cast<int>(n_splits);
  const int num_kb = (K + kBK - 1) / kBK;
  const int kb0 = static_cast<int>((static_cast<long long>(rank) * num_kb) / n_splits);
  const int kb1 = static_cast<int>((static_cast<long long>(rank + 1) * num_kb) / n_splits);
  const int count = kb1 - kb0;
  const uint32_t x_bytes = static_cast<uint32_t>(n_mma) * kSkRowBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSkStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kSkTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The weights are never written by the kernel before this one, so the
  // first stages' weight tiles are requested before waiting for it; the
  // activations (its output) after.
  const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
  const int early = count < kSkStages ? count : kSkStages;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < early; ++i) {
      mbar_arrive_expect_tx(&full[i], kSkWStage + x_bytes);
      tma_load_2d_hint(smem + i * kSkWStage, &tmap_w, &full[i], (kb0 + i) * kBK, n_blk * kSkRowsW, pol_w);
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < count; ++i) {
        const int stage = i % kSkStages;
        const uint32_t phase = static_cast<uint32_t>(i / kSkStages) & 1u;
        const int kx = (kb0 + i) * kBK;
        if (i >= early) {
          if (!mbar_wait(&empty[stage], phase ^ 1u)) break;
          mbar_arrive_expect_tx(&full[stage], kSkWStage + x_bytes);
          tma_load_2d_hint(smem + stage * kSkWStage, &tmap_w, &full[stage], kx, n_blk * kSkRowsW, pol_w);
        }
        tma_load_2d(smem + kSkXOff + stage * kSkXStage, &tmap_x, &full[stage], kx, 0);
        ++issued;
      }
      // the copies issued here have landed before the CTA goes on (only this
      // thread arms the full barriers: a stage's last fill completes its
      // phase exactly when its bytes are in)
      for (int i = issued - 1; i >= 0 && i >= issued - kSkStages; --i)
        mbar_wait(&full[i % kSkStages], static_cast<uint32_t>(i / kSkStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    for (int i = 0; i < count; ++i) {
      const int stage = i % kSkStages;
      const uint32_t phase = static_cast<uint32_t>(i / kSkStages) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase))) break;
      tc_fence_after();
      const uint32_t w_addr = smem_u32(smem + stage * kSkWStage);
      const uint32_t x_addr = smem_u32(smem + kSkXOff + stage * kSkXStage);
#pragma unroll
      for (int k = 0; k < kBK / kMmaK; ++k)
        tc_mma_warp<kTF32>(tmem_base, smem_desc_sw128(w_addr + k * 32), smem_desc_sw128(x_addr + k * 32), idesc,
                           (i | k) != 0 ? 1u : 0u);
      tc_commit_warp(&empty[stage]);  // frees the slot once these MMAs have read it
    }
    tc_commit_warp(done);  // arrives when every MMA issued above has completed
  }

  // ----------------------------------------------- partial D^T to shared
  // every lane waits; the outcome is warp-uniform so the .sync.aligned
  // tcgen05.ld below never runs divergent
  const bool have = __all_sync(0xffffffffu, mbar_wait(done, 0));
  tc_fence_after();
  float* red = reinterpret_cast<float*>(smem);  // [m][128] fp32 over the stage buffers
  const int n_local = warp * 32 + lane;          // this thread's weight row = TMEM lane
  if (have) {
    for (int c0 = 0; c0 < n_mma; c0 += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(c0), r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < M) red[(c0 + j) * kSkRowsW + n_local] = __uint_as_float(r[j]);
    }
  } else {
    for (int m = 0; m < M; ++m) red[m * kSkRowsW + n_local] = 0.f;
  }
  tc_fence_before();
  cluster_sync();  // every CTA's partial is written and visible to the cluster

  // ------------------------------------- reduce this CTA's slice, epilogue
  const int e4 = M * (kSkRowsW / 4);  // float4s in the [M][128] block
  const int per = (e4 + static_cast<int>(n_splits) - 1) / static_cast<int>(n_splits);
  const int lo = static_cast<int>(rank) * per;
  const int hi = min(e4, lo + per);
  const uint32_t red_addr = smem_u32(red);
  const bool vec_out = (N & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  for (int i = lo + static_cast<int>(threadIdx.x); i < hi; i += kSkThreads) {
    const uint32_t a = red_addr + static_cast<uint32_t>(i) * 16u;
    float4 acc = ld_shared_cluster_f4(mapa_shared(a, 0));
    for (uint32_t p = 1; p < n_splits; ++p) {
      const float4 t = ld_shared_cluster_f4(mapa_shared(a, p));
      acc.x += t.x;
      acc.y += t.y;
      acc.z += t.z;
      acc.w += t.w;
    }
    const int m = i / (kSkRowsW / 4);
    const int n = n_blk * kSkRowsW + (i % (kSkRowsW / 4)) * 4;
    if (n >= N) continue;
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    if (bias != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n + j < N) v[j] += __ldg(bias + n + j);
    }
    const size_t o = static_cast<size_t>(m) * N + n;
    if constexpr (kEpi == kEpiF32 || kEpi == kEpiResidF32) {
      float* of = static_cast<float*>(out) + o;
      if (vec_out && n + 3 < N) {
        float4 w = make_float4(v[0], v[1], v[2], v[3]);
        if constexpr (kEpi == kEpiResidF32) {
          const float4 old = *reinterpret_cast<const float4*>(of);
          w.x += old.x;
          w.y += old.y;
          w.z += old.z;
          w.w += old.w;
        }
        *reinterpret_cast<float4*>(of) = w;
      } else {
        for (int j = 0; j < 4 && n + j < N; ++j) of[j] = (kEpi == kEpiResidF32 ? of[j] : 0.f) + v[j];
      }
    } else {
      if constexpr (kEpi == kEpiGelu16) {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = gelu_fast(v[j]);
      }
      Out16* oh = static_cast<Out16*>(out) + o;
      if (vec_out && n + 3 < N) {
        uint2 p;
        p.x = pack2<Out16>(v[0], v[1]);
        p.y = pack2<Out16>(v[2], v[3]);
        *reinterpret_cast<uint2*>(oh) = p;
      } else {
        for (int j = 0; j < 4 && n + j < N; ++j) oh[j] = from_f32<Out16>(v[j]);
      }
    }
  }
  cluster_sync();  // the peers have read this CTA's partial
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSkTmemCols);
  }
}

bool skinny_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int rows, int cols,
                int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(cols) * elem_bytes};
  const uint32_t box[2] = {static_cast<uint32_t>(kSkRowBytes / elem_bytes), static_cast<uint32_t>(box_rows)};
  return encode_tensor_map_sw128(map, dt, 2, base, dims, strides, box);
}

template <int kEpi, int kOp>
int launch_skinny_impl(void* out, const void* A, const void* W, const float* bias, int M, int N, int K,
                       cudaStream_t s) {
  constexpr bool kTF32 = (kOp == kOpTF32);
  const int eb = kTF32 ? 4 : 2;
  const CUtensorMapDataType dt = kTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : (kOp == kOpF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  const int n_mma = (M + 15) / 16 * 16;
  CUtensorMap tw, tx;
  if (!skinny_map(&tw, W, dt, eb, N, K, kSkRowsW)) return GPT2_ERR_CUDA;
  if (!skinny_map(&tx, A, dt, eb, M, K, n_mma)) return GPT2_ERR_CUDA;
  auto kern = gemm_skinny_kernel<kEpi, kOp>;
  // per template instance and device: attributes, and whether clusters of
  // 16 (beyond the portable 8) can be resident
  static int max_splits[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits for its predecessor itself
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = kSkAlloc;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_splits[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSkAlloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    int ms = 8;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      attr[0].val.clusterDim.x = kSkMaxSplits;
      cfg.gridDim = dim3(kSkMaxSplits);
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) ms = kSkMaxSplits;
    }
    (void)cudaGetLastError();  // a refused query leaves no sticky error
    max_splits[dev] = ms;
  }
  const int n_blocks = (N + kSkRowsW - 1) / kSkRowsW;
  const int num_kb = (K + kSkRowBytes / eb - 1) / (kSkRowBytes / eb);
  // splits: a power of two, until about one CTA per SM, at least one K
  // block per split
  int splits = 1;
  while (splits * 2 <= max_splits[dev] && splits * 2 <= num_kb && n_blocks * splits < num_sms()) splits *= 2;
  attr[0].val.clusterDim.x = splits;
  cfg.gridDim = dim3(n_blocks * splits);
  cfg.numAttrs = pdl_on() ? 2 : 1;
  const uint32_t idesc = make_idesc(kOp == kOpF16 ? 0u : (kTF32 ? 2u : 1u), kSkRowsW, n_mma);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, tx, out, bias, M, N, K, n_mma, idesc);
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}

template <int kOp>
int launch_skinny_op(void* out, const void* A, const void* W, const float* bias, int M, int N, int K, int epi,
                     cudaStream_t s) {
  switch (epi) {
    case kEpiF32: return launch_skinny_impl<kEpiF32, kOp>(out, A, W, bias, M, N, K, s);
    case kEpiResidF32: return launch_skinny_impl<kEpiResidF32, kOp>(out, A, W, bias, M, N, K, s);
  }
  if constexpr (kOp != kOpTF32) {
    switch (epi) {
      case kEpiOut16: return launch_skinny_impl<kEpiOut16, kOp>(out, A, W, bias, M, N, K, s);
      case kEpiGelu16: return launch_skinny_impl<kEpiGelu16, kOp>(out, A, W, bias, M, N, K, s);
    }
  }
  return GPT2_ERR_UNSUPPORTED;
}

}  // namespace

int launch_gemm_skinny(void* out, const void* A, const void* W, const float* bias, int M, int N, int K, int epi,
                       int op, cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0) return GPT2_OK;
  if (M > kSkMaxRows) return GPT2_ERR_UNSUPPORTED;
  switch (op) {
    case kOpBF16: return launch_skinny_op<kOpBF16>(out, A, W, bias, M, N, K, epi, s);
    case kOpF16: return launch_skinny_op<kOpF16>(out, A, W, bias, M, N, K, epi, s);
    case kOpTF32: return launch_skinny_op<kOpTF32>(out, A, W, bias, M, N, K, epi, s);
  }
  return GPT2_ERR_UNSUPPORTED;
}

}  // namespace gpt2
