// gemm_tc.cu -- the five GEMM sites of the GPT-2 forward pass (QKV, attention
// projection, MLP up-projection, MLP down-projection, tied LM head) on the
// sm_103a tensor cores.
//
//   D[M, N] = A[M, K] * B[N, K]^T   (A: activations, B: a Linear weight
//                                     stored [out, in], both K-major)
//
// Design (persistent, warp-specialised, one CTA per SM).  For M > 128 the
// CTAs run as pairs (clusters of two): a pair owns a 256 x 256 tile, each
// CTA loads its 128 rows of A and one half (128 rows) of the B tile, and
// the even CTA issues the pair MMA (tcgen05 cta_group::2, M = 256) that
// writes each CTA's 128 rows into its own TMEM.  The pair form runs at the
// full tensor rate (a 256 x 256 x 16 instruction per ~130 cycles, measured)
// and halves the B bytes each SM loads.  Small M uses one CTA per 128 x 256
// tile.
//   warp 0      TMA producer: 128 x 128-byte A and 256 (single) or 128
//               (pair) x 128-byte B boxes (128-byte swizzle) into a 3-stage
//               (single) or 5-stage (pair) shared-memory ring;
//   warp 1      allocates 512 TMEM columns and (in a pair: the even CTA's)
//               issues tcgen05.mma (128 or 256 x 256 x 16 for bf16 or fp16
//               operands, x 8 for tf32, per instruction) into one of two
//               256-column fp32 TMEM accumulators; the warp runs the loop,
//               one elected lane issues;
//   warps 2-9   epilogue, two warps per TMEM lane quadrant, each on half of
//               the tile's columns: tcgen05.ld 32 columns of their 32 lanes,
//               add bias, apply GELU or add the residual (TMA-loaded), stage
//               in swizzled shared memory and TMA-store.  Eight warps, not
//               four: with four the epilogue of a tile took longer than its
//               MMAs (measured).  The LM-head epilogue also leaves, per row
//               and per 128 columns, the maximum and the sum of
//               exp(logit - maximum) over the real vocabulary, so that the
//               softmax needs one pass.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  Tiles are walked M-fastest, so that concurrently running CTAs share
// one weight tile (B) while the activation matrix (A) stays in L2, unless A
// is too large for L2 and B small (the MLP down-projection: A is 100 MB at
// 16 x 1024 tokens): then N-fastest, so that the few tiles that read one
// block of A run together and A crosses HBM once.
// Every wait is bounded (about one second); on a timeout the CTA records
// GPT2_DEVERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include <mutex>

#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kBM = 128;  // rows of A (and of D) per CTA
constexpr int kBN = 256;  // columns of D per tile
constexpr int kRowBytes = 128;  // one swizzle atom row: 64 bf16 or 32 fp32 of K
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, each on half the tile's columns
constexpr int kStageBufBytes = 32 * 128;  // an epilogue warp's output staging: 32 rows x 128 bytes
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;

// Shared-memory layout of a CTA, single (kPair false) or one of a pair.
template <bool kPair>
struct Layout {
  static constexpr int kStages = kPair ? 6 : 3;
  static constexpr int kBRows = kPair ? kBN / 2 : kBN;  // B rows this CTA loads per stage
  static constexpr int kAStageBytes = kBM * kRowBytes;
  static constexpr int kBStageBytes = kBRows * kRowBytes;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kStages * kAStageBytes;
  static constexpr int stg_off = b_off + kStages * kBStageBytes;
  static constexpr int bar_off = stg_off + kEpiWarps * kStageBufBytes;
  // barriers: full[S], empty[S], tmem_full[2], tmem_empty[2], res[kEpiWarps], drain
  static constexpr int n_bars = 2 * kStages + 4 + kEpiWarps + 1;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int total = misc_off + 16;
  static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};
static_assert(Layout<false>::alloc <= 232448 && Layout<true>::alloc <= 232448, "shared memory budget");

__host__ __device__ constexpr int gridDim_n(int N) { return (N + kBN - 1) / kBN; }
// LM-head softmax statistics per row: one (max, sum) per half tile (the
// columns one epilogue warp covers)
__host__ __device__ constexpr int stat_blocks(int N) { return 2 * gridDim_n(N); }

template <int kEpi, int kOp, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_out, const __grid_constant__ CUtensorMap tmap_res,
                   const float* __restrict__ bias, int M, int N, int K, int tiles_m, int num_tiles, int n_fast,
                   float2* __restrict__ row_stats, int V, int tiles_mn, int kb_per_split) {
  using L = Layout<kPair>;
  constexpr int kStages = L::kStages;
  constexpr int kAStageBytes = L::kAStageBytes;
  constexpr int kBStageBytes = L::kBStageBytes;
  constexpr int kTileM = kPair ? 2 * kBM : kBM;  // rows of a tile (a pair's or a CTA's)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tmem_full = bars + 2 * kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* res_bar = tmem_empty + 2;
  uint64_t* drain_bar = res_bar + kEpiWarps;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // a pair walks the tiles together: rank 0 or 1 within it, pair index
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int n_units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  constexpr bool kTF32 = (kOp == kOpTF32);
  using Out16 = typename std::conditional<kOp == kOpF16, __half, __nv_bfloat16>::type;
  constexpr int kElemBytes = kTF32 ? 4 : 2;
  constexpr int kBKElems = kRowBytes / kElemBytes;  // K elements per stage
  constexpr int kMmaK = 32 / kElemBytes;            // K per instruction (32 bytes)
  // operand format field: fp16 0, bf16 1 (kind::f16), tf32 2 (kind::tf32)
  constexpr uint32_t kIdesc = make_idesc(kOp == kOpF16 ? 0u : (kTF32 ? 2u : 1u), kTileM, kBN);
  const int num_kb = (K + kBKElems - 1) / kBKElems;
  // unit index -> (split of the K range, tile); tile -> (row block, column
  // block): M-fastest (concurrent tiles share a weight tile) or, with
  // n_fast, N-fastest (they share an activation block: for a large A and a
  // small B).  Without a K split there is one split and units are tiles.
  const int tiles_n = tiles_mn / tiles_m;
  auto tile_m = [&](int unit_) {
    const int tile = unit_ % tiles_mn;
    return n_fast ? tile / tiles_n : tile % tiles_m;
  };
  auto tile_n = [&](int unit_) {
    const int tile = unit_ % tiles_mn;
    return n_fast ? tile % tiles_n : tile / tiles_m;
  };
  auto kb_begin = [&](int unit_) { return (unit_ / tiles_mn) * kb_per_split; };
  auto kb_end = [&](int unit_) { return min(num_kb, (unit_ / tiles_mn + 1) * kb_per_split); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], kPair ? 2 : 1);  // pair: both producers arrive on the even CTA's barrier
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], kPair ? 2 * kEpiWarps : kEpiWarps);  // pair: both CTAs' epilogues
    }
    for (int i = 0; i < kEpiWarps; ++i) mbar_init(&res_bar[i], 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_out);
    if constexpr (kEpi == kEpiResidF32 || kEpi == kEpiGeluBwdF32 || kEpi == kEpiGeluDualF32)
      tma_prefetch_desc(&tmap_res);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();  // the peer's barriers are initialised before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // a programmatic dependent launch: the kernel ahead has finished
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0, fill_parity = 0;  // per stage: ever filled, parity of its last fill
      for (int tile = unit; tile < num_tiles && !*abort_flag; tile += n_units) {
        const int m_blk = tile_m(tile), n_blk = tile_n(tile);
        const int a_row = m_blk * kTileM + static_cast<int>(rank) * kBM;
        const int b_row = n_blk * kBN + static_cast<int>(rank) * L::kBRows;
        bool ok = true;
        for (int kb = kb_begin(tile); kb < kb_end(tile); ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            ok = false;
            break;
          }
          if constexpr (kPair) {  // both CTAs' bytes complete the even CTA's full barrier
            const uint32_t full_even = mapa_shared(smem_u32(&full[stage]), 0);
            mbar_arrive_expect_tx_cluster(full_even, kAStageBytes + kBStageBytes);
            tma_load_2d_pair(smem + L::a_off + stage * kAStageBytes, &tmap_a, full_even, kb * kBKElems, a_row);
            tma_load_2d_pair(smem + L::b_off + stage * kBStageBytes, &tmap_b, full_even, kb * kBKElems, b_row);
          } else {
            mbar_arrive_expect_tx(&full[stage], kAStageBytes + kBStageBytes);
            tma_load_2d_hint(smem + L::a_off + stage * kAStageBytes, &tmap_a, &full[stage], kb * kBKElems, a_row,
                             pol_a);
            tma_load_2d(smem + L::b_off + stage * kBStageBytes, &tmap_b, &full[stage], kb * kBKElems, b_row);
          }
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
      // Before the CTA may exit, the copies issued here must have landed:
      // single, only this thread arms the full barriers, so the phase of a
      // stage's last fill completes exactly when its bytes have landed; in a
      // pair the full barriers are the even CTA's, so wait instead for the
      // MMAs that consumed the last fill to release the slot (immediate in
      // the normal case).
      for (int s = 0; s < kStages; ++s)
        if ((filled >> s) & 1u) mbar_wait(kPair ? &empty[s] : &full[s], (fill_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (rank == 0) {  // in a pair the even CTA issues for both; the warp runs the loop, one lane issues
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = unit; tile < num_tiles && __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
           tile += n_units, ++local) {  // one read for the whole warp: it must not split
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tmem_empty[acc], acc_phase ^ 1))) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        bool ok = true;
        const int kb0 = kb_begin(tile);
        for (int kb = kb0; kb < kb_end(tile); ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + L::a_off + stage * kAStageBytes);
          const uint32_t b_addr = smem_u32(smem + L::b_off + stage * kBStageBytes);
#pragma unroll
          for (int k = 0; k < kBKElems / kMmaK; ++k) {
            if constexpr (kPair)
              tc_mma_pair_warp<kTF32>(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32),
                                      kIdesc, (kb != kb0 || k != 0) ? 1u : 0u);
            else
              tc_mma_warp<kTF32>(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), kIdesc,
                                 (kb != kb0 || k != 0) ? 1u : 0u);
          }
          // frees the smem slot (in both CTAs of a pair) once these MMAs have read it
          if constexpr (kPair)
            tc_commit_pair_warp(&empty[stage], 3);
          else
            tc_commit_warp(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if constexpr (kPair)
          tc_commit_pair_warp(&tmem_full[acc], 3);
        else
          tc_commit_warp(&tmem_full[acc]);
      }
      // every MMA issued above has completed once this commit arrives
      if constexpr (kPair)
        tc_commit_pair_warp(drain_bar, 1);
      else
        tc_commit_warp(drain_bar);
      mbar_wait(drain_bar, 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2;            // epilogue warp index 0..7
    const int quad = warp & 3;          // TMEM lane quadrant this warp may access
    const int row_in_tile = quad * 32;  // tile rows [row_in_tile, row_in_tile + 32)
    const int col_half = ew >> 2;       // tile columns [128 col_half, 128 col_half + 128)
    uint8_t* stg = smem + L::stg_off + ew * kStageBufBytes;
    uint32_t res_phase = 0;  // parity of this warp's next residual load
    // The bias of this warp's 128 columns of a tile, lane l holding columns
    // 4l .. 4l + 3 (zero past N), loaded a tile ahead and handed out by
    // shuffles: with most of the SM's shared memory in use the L1 cache is
    // small, and a load per chunk would wait on L2 every time.
    auto load_bias = [&](int tile) -> float4 {
      float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bias != nullptr && tile < num_tiles) {
        const int c = tile_n(tile) * kBN + col_half * (kBN / 2) + 4 * lane;
        if (c + 3 < N) {
          r = __ldg(reinterpret_cast<const float4*>(bias + c));
        } else {
          if (c < N) r.x = __ldg(bias + c);
          if (c + 1 < N) r.y = __ldg(bias + c + 1);
          if (c + 2 < N) r.z = __ldg(bias + c + 2);
        }
      }
      return r;
    };
    float4 bias_cur = load_bias(unit);
    int local = 0;
    for (int tile = unit; tile < num_tiles && __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
         tile += n_units, ++local) {  // one read for the whole warp: it must not split
      const int m_blk = tile_m(tile), n_blk = tile_n(tile);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const float4 bias_next = load_bias(tile + n_units);
      // every lane waits; the outcome is made warp-uniform so that the
      // .sync.aligned tcgen05 instructions below never run divergent
      if (!__all_sync(0xffffffffu, mbar_wait(&tmem_full[acc], acc_phase))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int m0 = m_blk * kTileM + static_cast<int>(rank) * kBM + row_in_tile;
      const int n0 = n_blk * kBN;
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(row_in_tile) << 16) + static_cast<uint32_t>(acc * kBN);
      constexpr bool kOutF32 = (kEpi == kEpiF32 || kEpi == kEpiResidF32 || kEpi == kEpiLogits ||
                                kEpi == kEpiGeluBwdF32 || kEpi == kEpiGeluDualF32);
      constexpr bool kAux = (kEpi == kEpiResidF32 || kEpi == kEpiGeluBwdF32);  // reads a tile of tmap_res
      constexpr int kChunkCols = kOutF32 ? 32 : 64;  // 128 bytes of output per row
      // logits epilogue: this row's running max and sum of exp over the
      // tile's columns below V
      float run_m = -INFINITY, run_s = 0.f;
      // a warp whose 32 rows all lie past M (a few activation rows, as the
      // decode step's LM head has) has nothing to write: it only frees the
      // accumulator
      const bool live = m0 < M;
#pragma unroll 1
      for (int ch = col_half * (kBN / kChunkCols / 2); live && ch < (col_half + 1) * (kBN / kChunkCols / 2); ++ch) {
        const int col0 = n0 + ch * kChunkCols;
        bool ok = true;
        if constexpr (kAux) {  // the residual (or GELU input) tile into the staging buffer
          if (lane == 0) {
            bulk_wait_group_read<0>();  // the previous store has read the buffer
            mbar_arrive_expect_tx(&res_bar[ew], kStageBufBytes);
            tma_load_3d(stg, &tmap_res, &res_bar[ew], col0, m0, 0);
          }
        }
        float v[kChunkCols];
        {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_base + ch * kChunkCols, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          if constexpr (kChunkCols == 64) {
            tmem_ld_32x32b_x32(t_base + ch * kChunkCols + 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[32 + j] = __uint_as_float(r[j]);
          }
        }
        if (bias != nullptr) {
          const int src0 = (ch * kChunkCols - col_half * (kBN / 2)) / 4;  // lane holding the chunk's column 0
#pragma unroll
          for (int j = 0; j < kChunkCols / 4; ++j) {
            v[4 * j] += __shfl_sync(0xffffffffu, bias_cur.x, src0 + j);
            v[4 * j + 1] += __shfl_sync(0xffffffffu, bias_cur.y, src0 + j);
            v[4 * j + 2] += __shfl_sync(0xffffffffu, bias_cur.z, src0 + j);
            v[4 * j + 3] += __shfl_sync(0xffffffffu, bias_cur.w, src0 + j);
          }
        }
        if constexpr (kEpi == kEpiLogits) {
          // (max, sum of exp) over the chunk's columns below V, folded into
          // the row's running pair.  Four independent max and sum chains
          // (one long chain per thread left the epilogue slower than the
          // MMAs), exp(x - m) as exp2(x log2e - m log2e).
          constexpr float kLog2e = 1.4426950408889634f;
          const bool full = col0 + 32 <= V;  // the same for the whole warp
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (full || col0 + j < V) m4[j & 3] = fmaxf(m4[j & 3], v[j]);
          const float cmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          if (cmax != -INFINITY) {
            const float m_new = fmaxf(run_m, cmax);
            const float mb = m_new * kLog2e;
            float s4[4] = {run_s * exp2_approx(run_m * kLog2e - mb), 0.f, 0.f, 0.f};  // 0 while run_m is -inf
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (full || col0 + j < V) s4[j & 3] += exp2_approx(fmaf(v[j], kLog2e, -mb));
            run_m = m_new;
            run_s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
          }
        }
        // Stage the chunk (32 rows x 128 bytes, 128-byte swizzle) in this
        // warp's buffer and TMA-store it.  One buffer per warp: the store of
        // the previous chunk has had this chunk's loads and math to read it.
        if (!kAux && lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        const int sw = lane & 7;
        uint8_t* my_row = stg + lane * 128;
        if constexpr (kOutF32) {
          if constexpr (kAux) {
            ok = __all_sync(0xffffffffu, mbar_wait(&res_bar[ew], res_phase));
            res_phase ^= 1u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 old = *reinterpret_cast<const float4*>(my_row + ((j ^ sw) << 4));
              if constexpr (kEpi == kEpiResidF32) {
                v[4 * j] += old.x;
                v[4 * j + 1] += old.y;
                v[4 * j + 2] += old.z;
                v[4 * j + 3] += old.w;
              } else {  // the gradient through the GELU whose input is old
                v[4 * j] *= gelu_grad(old.x);
                v[4 * j + 1] *= gelu_grad(old.y);
                v[4 * j + 2] *= gelu_grad(old.z);
                v[4 * j + 3] *= gelu_grad(old.w);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(my_row + ((j ^ sw) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float a[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              a[e] = v[8 * j + e];
              if constexpr (kEpi == kEpiGelu16) a[e] = gelu_fast(a[e]);
            }
            uint4 p;
            p.x = pack2<Out16>(a[0], a[1]);
            p.y = pack2<Out16>(a[2], a[3]);
            p.z = pack2<Out16>(a[4], a[5]);
            p.w = pack2<Out16>(a[6], a[7]);
            *reinterpret_cast<uint4*>(my_row + ((j ^ sw) << 4)) = p;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmap_out, stg, col0, m0, tile / tiles_mn);  // the split's slice of the output
          bulk_commit_group();
        }
        if constexpr (kEpi == kEpiGeluDualF32) {
          // the chunk's GELU, the second output, through the same buffer
          // once the store above has read it
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(my_row + ((j ^ sw) << 4)) =
                make_float4(gelu_exact(v[4 * j]), gelu_exact(v[4 * j + 1]), gelu_exact(v[4 * j + 2]),
                            gelu_exact(v[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmap_res, stg, col0, m0, 0);
            bulk_commit_group();
          }
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
      if constexpr (kEpi == kEpiLogits) {
        const int row = m0 + lane;
        if (row < M) row_stats[static_cast<size_t>(row) * stat_blocks(N) + 2 * n_blk + col_half] = make_float2(run_m, run_s);
      }
      // this warp is done reading the accumulator
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[acc]), 0));  // the even CTA's barrier
        else
          mbar_arrive(&tmem_empty[acc]);
      }
      bias_cur = bias_next;
    }
    if (lane == 0) bulk_wait_group<0>();  // stores complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();  // neither CTA leaves while the pair MMAs may read its shared memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over a row-major [rows, cols] matrix with a box of
// box_cols x box_rows and the 128-byte swizzle (box_cols * elem = 128).
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int rows, int cols,
              int box_cols, int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(cols) * elem_bytes};
  const uint32_t box[2] = {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows)};
  return encode_tensor_map_sw128(map, dt, 2, base, dims, strides, box);
}

// The output: `depth` slices of [rows][cols] one after another (the slices
// of a K split; depth 1 otherwise)
bool make_out_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int rows, int cols,
                  int depth, int box_cols, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), static_cast<uint64_t>(depth)};
  const uint64_t strides[2] = {static_cast<uint64_t>(cols) * elem_bytes,
                               static_cast<uint64_t>(rows) * cols * elem_bytes};
  const uint32_t box[3] = {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows), 1};
  return encode_tensor_map_sw128(map, dt, 3, base, dims, strides, box);
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  const CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tensor_map_sw128(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tensor_map(map, dt, rank, base, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

namespace {

template <int kEpi, int kOp, bool kPair>
int launch_impl(void* out, const void* A, const void* B, const float* bias, int M, int N, int K, cudaStream_t s,
                float2* row_stats, int V, int splits = 1, const float* resid = nullptr) {
  using L = Layout<kPair>;
  CUtensorMap ta, tb, to, tr;
  constexpr bool kTF32 = (kOp == kOpTF32);
  const CUtensorMapDataType dt16 =
      kOp == kOpF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType dt_in = kTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt16;
  const int eb = kTF32 ? 4 : 2;
  const int bk = kRowBytes / eb;
  constexpr bool kOutF32 = (kEpi == kEpiF32 || kEpi == kEpiResidF32 || kEpi == kEpiLogits ||
                            kEpi == kEpiGeluBwdF32 || kEpi == kEpiGeluDualF32);
  if (!make_map(&ta, A, dt_in, eb, M, K, bk, kBM)) return GPT2_ERR_CUDA;
  if (!make_map(&tb, B, dt_in, eb, N, K, bk, L::kBRows)) return GPT2_ERR_CUDA;
  const int num_kb = (K + bk - 1) / bk;
  const int kb_per_split = (num_kb + splits - 1) / splits;
  splits = (num_kb + kb_per_split - 1) / kb_per_split;  // no empty split
  if (kOutF32) {
    if (!make_out_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N, splits, 32, 32)) return GPT2_ERR_CUDA;
  } else {
    if (!make_out_map(&to, out, dt16, 2, M, N, splits, 64, 32)) return GPT2_ERR_CUDA;
  }
  // the tile source of the epilogues that read one: `resid` when given,
  // else the output itself (the residual epilogue's out += ...)
  tr = to;
  if ((kEpi == kEpiResidF32 || kEpi == kEpiGeluBwdF32 || kEpi == kEpiGeluDualF32) && resid != nullptr &&
      resid != out)
    if (!make_out_map(&tr, resid, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N, 1, 32, 32)) return GPT2_ERR_CUDA;
  constexpr int kTileM = kPair ? 2 * kBM : kBM;
  const int tiles_m = (M + kTileM - 1) / kTileM;
  const int tiles_n = (N + kBN - 1) / kBN;
  const int tiles_mn = tiles_m * tiles_n;
  const int num_tiles = tiles_mn * splits;  // units: (split, tile)
  const size_t a_bytes = static_cast<size_t>(M) * K * eb, b_bytes = static_cast<size_t>(N) * K * eb;
  const int n_fast = (a_bytes > (48u << 20) && b_bytes < (32u << 20)) ? 1 : 0;
  auto kern = gemm_tc_kernel<kEpi, kOp, kPair>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::alloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits for its predecessor itself
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // per template instance and device: the shared-memory attribute and how
  // many CTAs (or pairs) can be resident at once
  static int resident[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (resident[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    int n = kPair ? num_sms() / 2 : num_sms();
    if (kPair) {
      cfg.gridDim = dim3(2 * n);
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return note_cuda_error(e);
      if (clusters > 0 && clusters < n) n = clusters;
    }
    resident[dev] = n;
  }
  const int units = num_tiles < resident[dev] ? num_tiles : resident[dev];
  cfg.gridDim = dim3(kPair ? 2 * units : units);
  cfg.numAttrs = pdl_on() ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, to, tr, bias, M, N, K, tiles_m, num_tiles, n_fast,
                                           row_stats, V, tiles_mn, kb_per_split);
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}

// out = the sum of the `splits` slices of part ([splits][n] fp32), in slice
// order (the result does not depend on timing); vec: 16-byte accesses
__global__ void splitk_sum_kernel(float* __restrict__ out, const float* __restrict__ part, long long n, int splits,
                                  int vec) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (vec) {
    const long long n4 = n / 4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4; i += stride) {
      float4 acc = __ldg(reinterpret_cast<const float4*>(part) + i);
      for (int sp = 1; sp < splits; ++sp) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(part + sp * n) + i);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      reinterpret_cast<float4*>(out)[i] = acc;
    }
  } else {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride) {
      float acc = part[i];
      for (int sp = 1; sp < splits; ++sp) acc += part[sp * n + i];
      out[i] = acc;
    }
  }
}

template <int kEpi, int kOp>
int launch_typed(void* out, const void* A, const void* B, const float* bias, int M, int N, int K, cudaStream_t s,
                 float2* row_stats = nullptr, int V = 0, const float* resid = nullptr) {
  if (M > kBM) return launch_impl<kEpi, kOp, true>(out, A, B, bias, M, N, K, s, row_stats, V, 1, resid);
  return launch_impl<kEpi, kOp, false>(out, A, B, bias, M, N, K, s, row_stats, V, 1, resid);
}

}  // namespace

int launch_gemm_tc(void* out, const void* A, const void* B, const float* bias, int M, int N, int K, int epi, int op,
                   cudaStream_t s, const float* resid) {
  if (M <= 0 || N <= 0 || K <= 0) return GPT2_OK;
  const bool two_tensor = epi == kEpiGeluBwdF32 || epi == kEpiGeluDualF32;  // resid required
  if (resid != nullptr && resid != out && (epi != kEpiResidF32 || M <= kSkinnyMaxRows) && !two_tensor)
    return GPT2_ERR_UNSUPPORTED;
  if (two_tensor && (resid == nullptr || resid == out || M <= kSkinnyMaxRows || op != kOpTF32))
    return GPT2_ERR_UNSUPPORTED;
  if (M <= kSkinnyMaxRows) return launch_gemm_skinny(out, A, B, bias, M, N, K, epi, op, s);
  switch (op) {
    case kOpBF16:
      switch (epi) {
        case kEpiF32: return launch_typed<kEpiF32, kOpBF16>(out, A, B, bias, M, N, K, s);
        case kEpiOut16: return launch_typed<kEpiOut16, kOpBF16>(out, A, B, bias, M, N, K, s);
        case kEpiGelu16: return launch_typed<kEpiGelu16, kOpBF16>(out, A, B, bias, M, N, K, s);
        case kEpiResidF32: return launch_typed<kEpiResidF32, kOpBF16>(out, A, B, bias, M, N, K, s, nullptr, 0, resid);
      }
      break;
    case kOpF16:
      switch (epi) {
        case kEpiF32: return launch_typed<kEpiF32, kOpF16>(out, A, B, bias, M, N, K, s);
        case kEpiOut16: return launch_typed<kEpiOut16, kOpF16>(out, A, B, bias, M, N, K, s);
        case kEpiGelu16: return launch_typed<kEpiGelu16, kOpF16>(out, A, B, bias, M, N, K, s);
        case kEpiResidF32: return launch_typed<kEpiResidF32, kOpF16>(out, A, B, bias, M, N, K, s, nullptr, 0, resid);
      }
      break;
    case kOpTF32:
      switch (epi) {
        case kEpiF32: return launch_typed<kEpiF32, kOpTF32>(out, A, B, bias, M, N, K, s);
        case kEpiResidF32: return launch_typed<kEpiResidF32, kOpTF32>(out, A, B, bias, M, N, K, s, nullptr, 0, resid);
        case kEpiGeluBwdF32:
          return launch_typed<kEpiGeluBwdF32, kOpTF32>(out, A, B, bias, M, N, K, s, nullptr, 0, resid);
        case kEpiGeluDualF32:
          return launch_typed<kEpiGeluDualF32, kOpTF32>(out, A, B, bias, M, N, K, s, nullptr, 0, resid);
      }
      break;
  }
  return GPT2_ERR_UNSUPPORTED;
}

int splitk_choose(int M, int N, int K, int op, size_t partial_floats) {
  if (M <= kBM || M <= kSkinnyMaxRows) return 1;  // the pair kernel only
  const int bk = kRowBytes / (op == kOpTF32 ? 4 : 2);
  const int num_kb = (K + bk - 1) / bk;
  const int tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + kBN - 1) / kBN);
  const int resident = num_sms() / 2;  // CTA pairs
  // fewest rounds x k-blocks per split, each split at least 8 k-blocks,
  // within the partial buffer
  int best = 1;
  long long best_cost = static_cast<long long>((tiles + resident - 1) / resident) * num_kb;
  for (int sp = 2; sp <= 32 && sp * 8 <= num_kb; ++sp) {
    if (static_cast<size_t>(sp) * M * N > partial_floats) break;
    const int kbps = (num_kb + sp - 1) / sp;
    const long long cost = static_cast<long long>((tiles * sp + resident - 1) / resident) * kbps;
    if (cost < best_cost) {
      best = sp;
      best_cost = cost;
    }
  }
  return best;
}

int launch_gemm_tc_splitk(float* out, float* partials, size_t partial_floats, const void* A, const void* B, int M,
                          int N, int K, int op, cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0) return GPT2_OK;
  const int splits = splitk_choose(M, N, K, op, partial_floats);
  if (splits == 1) return launch_gemm_tc(out, A, B, nullptr, M, N, K, kEpiF32, op, s);
  int rc = GPT2_ERR_UNSUPPORTED;
  switch (op) {
    case kOpBF16: rc = launch_impl<kEpiF32, kOpBF16, true>(partials, A, B, nullptr, M, N, K, s, nullptr, 0, splits); break;
    case kOpF16: rc = launch_impl<kEpiF32, kOpF16, true>(partials, A, B, nullptr, M, N, K, s, nullptr, 0, splits); break;
    case kOpTF32: rc = launch_impl<kEpiF32, kOpTF32, true>(partials, A, B, nullptr, M, N, K, s, nullptr, 0, splits); break;
  }
  if (rc != GPT2_OK) return rc;
  const long long n = static_cast<long long>(M) * N;
  const int vec = (n % 4 == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(partials) & 15u) == 0)
                      ? 1
                      : 0;
  const long long work = vec ? n / 4 : n;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  const long long want = (work + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  splitk_sum_kernel<<<blocks, 256, 0, s>>>(out, partials, n, splits, vec);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}

int launch_gemm_logits(float* logits, float2* row_stats, const void* A, const void* B, int M, int N, int K, int V,
                       int op, cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0) return GPT2_OK;
  switch (op) {
    case kOpBF16: return launch_typed<kEpiLogits, kOpBF16>(logits, A, B, nullptr, M, N, K, s, row_stats, V);
    case kOpF16: return launch_typed<kEpiLogits, kOpF16>(logits, A, B, nullptr, M, N, K, s, row_stats, V);
    case kOpTF32: return launch_typed<kEpiLogits, kOpTF32>(logits, A, B, nullptr, M, N, K, s, row_stats, V);
  }
  return GPT2_ERR_UNSUPPORTED;
}

int logits_stat_blocks(int N) { return stat_blocks(N); }

}  // namespace gpt2
