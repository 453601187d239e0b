// attention.cu -- causal multi-head attention of the GPT-2 forward pass.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); it is computed the Algorithm 1 way: key/value tiles stream
// through shared memory while each query row keeps a running maximum, a
// running sum and an unnormalised output, so the T x T score matrix never
// exists.  Key tiles wholly after a query tile are never visited (causal
// tile skipping); only the diagonal tile is masked.  Heads are read in place
// from the fused QKV buffer [B, T, 3C] (query, key, value column blocks, head
// h = columns h*hs .. h*hs+hs-1 of each), and the output is written straight
// into [B, T, C]: no permute or unpermute pass.
//
//   attn_tc_kernel      tensor cores (mma.sync m16n8k16 on bf16 or fp16
//                       operands, fp32 accumulate), head size 16 or 32, 64
//                       query rows per block (head size 64, GPT-2's, runs
//                       on the tcgen05 kernel of attention_tc.cu);
//   attn_f32_kernel     fp32 CUDA cores, reference-grade (GPT2_FP32 mode);
//   decode_attn_kernel  one query per sequence against the KV cache, one
//                       block per (head, sequence).
#include "kernels.cuh"

namespace gpt2 {
namespace {

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d += a * b, m16n8k16, 16-bit inputs of type T (bf16 or fp16), fp32 accumulators
template <typename T>
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------- bf16 tensor-core kernel
constexpr int kBQ = 64;    // query rows per block (16 per warp)
constexpr int kBKV = 64;   // keys per tile
constexpr int kAttnThreads = 128;

// A tile is 64 rows of HS bf16 (HS * 2 bytes, HS / 8 chunks of 16 bytes);
// chunk c of row r is stored at chunk (c ^ (r mod chunks)) so that the eight
// row addresses of an ldmatrix fall in distinct banks.
template <int HS>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  constexpr int kChunks = HS / 8;
  return static_cast<uint32_t>(row * (HS * 2) + ((chunk ^ (row & (kChunks - 1))) << 4));
}

// Loads rows [row0, row0+64) (row index = token t of sequence b) of the
// HS-wide column block starting at `col` of qkv into a swizzled tile; rows
// at or beyond T are zero-filled.
template <int HS>
__device__ __forceinline__ void load_tile(uint8_t* tile, const uint16_t* qkv, int b, int T, int C3, int col,
                                          int row0) {
  constexpr int kChunks = HS / 8;
  for (int idx = threadIdx.x; idx < kBKV * kChunks; idx += kAttnThreads) {
    const int r = idx / kChunks, c = idx % kChunks;
    const int t = row0 + r;
    const bool valid = t < T;
    const uint16_t* src = qkv + (static_cast<size_t>(b) * T + (valid ? t : 0)) * C3 + col + c * 8;
    cp_async16(tile + swz<HS>(r, c), src, valid);
  }
}

template <int HS, typename T16, bool kOut16>
__global__ void __launch_bounds__(kAttnThreads) attn_tc_kernel(void* __restrict__ out, const uint16_t* __restrict__ qkv,
                                                               int T, int C, float scale_log2) {
  constexpr int kKS = HS / 16;  // k-steps of Q K^T over the head dimension
  constexpr int kDT = HS / 8;   // 8-wide output column tiles
  __shared__ __align__(128) uint8_t q_s[kBQ * HS * 2];
  __shared__ __align__(128) uint8_t k_s[2][kBKV * HS * 2];
  __shared__ __align__(128) uint8_t v_s[2][kBKV * HS * 2];

  const int n_qt = gridDim.x;
  const int qt = n_qt - 1 - blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int C3 = 3 * C;
  const int q0 = qt * kBQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;

  load_tile<HS>(q_s, qkv, b, T, C3, h * HS, q0);
  load_tile<HS>(k_s[0], qkv, b, T, C3, C + h * HS, 0);
  load_tile<HS>(v_s[0], qkv, b, T, C3, 2 * C + h * HS, 0);
  cp_async_commit();

  float o[kDT][4];
#pragma unroll
  for (int i = 0; i < kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  uint32_t qf[kKS][4];

  const int row_w = warp * 16;  // this warp's first query row in the tile
  for (int j = 0; j <= qt; ++j) {
    const int buf = j & 1;
    if (j < qt) {  // prefetch the next key/value tile
      load_tile<HS>(k_s[buf ^ 1], qkv, b, T, C3, C + h * HS, (j + 1) * kBKV);
      load_tile<HS>(v_s[buf ^ 1], qkv, b, T, C3, 2 * C + h * HS, (j + 1) * kBKV);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        const int r = row_w + (lane & 15);
        const int c = ks * 2 + (lane >> 4);
        ldsm_x4(smem_u32(q_s) + swz<HS>(r, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    // S = Q K^T for this warp's 16 rows and the tile's 64 keys
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    const uint32_t kb = smem_u32(k_s[buf]);
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<HS>(key, c), b0, b1, b2, b3);
        mma16<T16>(s[2 * np], qf[ks], b0, b1);
        mma16<T16>(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
    // scale into log2 units and mask the diagonal tile
    const bool diag = (j == qt);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * scale_log2;
        if (diag) {
          const int key = j * kBKV + nt * 8 + 2 * tig + (e & 1);
          const int qrow = q0 + row_w + g + ((e >> 1) << 3);
          if (key > qrow || key >= T) x = -INFINITY;
        }
        s[nt][e] = x;
      }
    }
    // online softmax: rows g (e = 0, 1) and g + 8 (e = 2, 3)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * r], s[nt][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_r[r], mx);
      const float alpha = exp2_fast(m_r[r] - m_new);  // 0 on the first tile (m = -inf)
      m_r[r] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float p0 = exp2_fast(s[nt][2 * r] - m_new);
        const float p1 = exp2_fast(s[nt][2 * r + 1] - m_new);
        s[nt][2 * r] = p0;
        s[nt][2 * r + 1] = p1;
        sum += p0 + p1;
      }
      l_r[r] = l_r[r] * alpha + sum;
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        o[dt][2 * r] *= alpha;
        o[dt][2 * r + 1] *= alpha;
      }
    }
    // O += P V: P's accumulator layout is the A-operand layout of k-steps
    const uint32_t vb = smem_u32(v_s[buf]);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t pa[4];
      pa[0] = pack2<T16>(s[2 * ks][0], s[2 * ks][1]);
      pa[1] = pack2<T16>(s[2 * ks][2], s[2 * ks][3]);
      pa[2] = pack2<T16>(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      pa[3] = pack2<T16>(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int dp = 0; dp < kDT / 2; ++dp) {
        const int key = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<HS>(key, c), b0, b1, b2, b3);
        mma16<T16>(o[2 * dp], pa, b0, b1);
        mma16<T16>(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // this buffer is refilled by the next iteration's prefetch
  }
  // normalise and store rows g and g + 8
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_r[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const float inv = 1.0f / l;
    const int t = q0 + row_w + g + 8 * r;
    if (t >= T) continue;
    const size_t base = (static_cast<size_t>(b) * T + t) * C + h * HS;
#pragma unroll
    for (int dt = 0; dt < kDT; ++dt) {
      const int d = dt * 8 + 2 * tig;
      const float x0 = o[dt][2 * r] * inv, x1 = o[dt][2 * r + 1] * inv;
      if constexpr (kOut16) {
        *reinterpret_cast<uint32_t*>(reinterpret_cast<T16*>(out) + base + d) = pack2<T16>(x0, x1);
      } else {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(out) + base + d) = make_float2(x0, x1);
      }
    }
  }
}

// -------------------------------------------------- fp32 reference kernel
// One thread per query row, 64 rows per block; key/value tiles of 64 rows
// in shared memory; exact expf; one key at a time with the running max.
template <int HS>
__global__ void __launch_bounds__(64) attn_f32_kernel(float* __restrict__ out, const float* __restrict__ qkv, int T,
                                                      int C, float scale) {
  __shared__ float k_s[64][HS];
  __shared__ float v_s[64][HS];
  const int qt = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int C3 = 3 * C;
  const int t = qt * 64 + threadIdx.x;
  const bool active = t < T;
  float q[HS], o[HS];
  const float* qrow = qkv + (static_cast<size_t>(b) * T + (active ? t : 0)) * C3 + h * HS;
#pragma unroll
  for (int d = 0; d < HS; ++d) {
    q[d] = qrow[d];
    o[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j0 = 0; j0 <= qt * 64; j0 += 64) {
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * HS; i += 64) {
      const int r = i / HS, d = i % HS;
      const int key = j0 + r;
      const size_t base = (static_cast<size_t>(b) * T + (key < T ? key : 0)) * C3 + h * HS + d;
      k_s[r][d] = key < T ? qkv[base + C] : 0.f;
      v_s[r][d] = key < T ? qkv[base + 2 * C] : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < 64; ++r) {
      const int key = j0 + r;
      if (key > t || key >= T) break;
      float dot = 0.f;
#pragma unroll
      for (int d = 0; d < HS; ++d) dot = fmaf(q[d], k_s[r][d], dot);
      const float sc = dot * scale;
      if (sc > m) {
        const float a = expf(m - sc);  // 0 when m = -inf
        l = l * a + 1.f;
#pragma unroll
        for (int d = 0; d < HS; ++d) o[d] = o[d] * a + v_s[r][d];
        m = sc;
      } else {
        const float p = expf(sc - m);
        l += p;
#pragma unroll
        for (int d = 0; d < HS; ++d) o[d] = fmaf(p, v_s[r][d], o[d]);
      }
    }
  }
  if (!active) return;
  const float inv = 1.f / l;
  float* orow = out + (static_cast<size_t>(b) * T + t) * C + h * HS;
#pragma unroll
  for (int d = 0; d < HS; ++d) orow[d] = o[d] * inv;
}

// ------------------------------------------------------------- decode
// One CTA of kDecWarps warps per (head, sequence).  A warp walks chunks of
// the cache (chunk w, w + kDecWarps, ...) keeping a running maximum, sum and
// unnormalised output (the online softmax of FlashAttention's Algorithm 1
// with a single query row).  Each K or V row is read by kLPR lanes with
// 16-byte loads, kRPI rows per warp instruction (coalesced), and a chunk's
// K and V loads are all issued before any is used.  At the end the CTA
// merges its warps' (maximum, sum, output) in shared memory and writes the
// head's output row: one launch, no scratch.  The token's own key and value
// (position pos) are read from the QKV row, and the block also appends them
// to the cache for the steps that follow.
//
// Cache rows are found through KVRows: a dense cache [B][NH][maxT][hs] per
// layer and K/V half, or a paged pool [num_blocks][NH][block][hs] whose
// block of position p of sequence b is table[b][p / block] (the block-table
// layout of a paged KV cache).  Positions come from `pos` (all sequences
// at one position) or, when pos_arr is given, per sequence from it.
constexpr int kDecWarps = 4;       // warps computing; one more issues the copies
constexpr int kDecStages = 8;      // chunks of the cache in shared memory
constexpr int kDecStageBytes = 8192;  // a chunk's K rows, then its V rows (4 KB each)
constexpr int kDecSmem = kDecStages * kDecStageBytes + 2 * kDecStages * 8;
// chunk c goes to warp c % kDecWarps and stage c % kDecStages: with the
// stages a multiple of the warps, the chunks that share a stage share a
// warp too, so no warp waits on a stage's barrier more than one phase ahead
// of the fill it needs (a waiter two phases ahead would pass at once)
static_assert(kDecStages % kDecWarps == 0, "stages per warp");

template <typename E, typename OutT, int HS>
__global__ void __launch_bounds__(32 * (kDecWarps + 1))
    decode_attn_kernel(OutT* __restrict__ out, const E* __restrict__ qkv, E* __restrict__ kcache,
                       E* __restrict__ vcache, int C, int NH, int pos_all, const int* __restrict__ pos_arr,
                       KVRows rows, float scale_log2) {
  constexpr int kPer = 16 / static_cast<int>(sizeof(E));  // elements per 16-byte load
  constexpr int kLPR = HS / kPer;                          // lanes per K or V row
  constexpr int kRPI = 32 / kLPR;                          // rows per warp instruction
  constexpr int kIt = 8;                                   // instructions per chunk (each of K, V)
  constexpr int kChunk = kIt * kRPI;                       // positions per chunk
  constexpr int kRowBytes = HS * static_cast<int>(sizeof(E));
  static_assert(kLPR >= 1 && kLPR <= 32 && 32 % kLPR == 0, "head size and element type");
  static_assert(kChunk * kRowBytes * 2 == kDecStageBytes, "a chunk's K and V fill a stage");
  extern __shared__ __align__(16) uint8_t dec_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(dec_smem + kDecStages * kDecStageBytes);
  uint64_t* empty = full + kDecStages;
  __shared__ float m_s[kDecWarps], l_s[kDecWarps];
  __shared__ float o_s[kDecWarps][HS];
  __shared__ int tbl_s[kMaxBlocksPerSeq];  // this sequence's block table (paged layout)
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / kLPR;   // row of an instruction this lane reads
  const int dg = lane % kLPR;  // its dimensions dg * kPer .. dg * kPer + kPer - 1
  // the caller's positions and block table are inputs of the step, written
  // before its first kernel: they may be read before the wait below
  const int pos = pos_arr != nullptr ? __ldg(pos_arr + b) : pos_all;
  const bool pos_ok = pos >= 0 && pos < rows.capacity;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(&full[i], 1u);
      mbar_init(&empty[i], 1u);
    }
    fence_barrier_init();
  }
  if (rows.table != nullptr && pos_ok) {
    for (int i = threadIdx.x; i <= (pos >> rows.lbs); i += blockDim.x) {
      int blk = __ldg(rows.table + static_cast<size_t>(b) * rows.max_blocks + i);
      if (blk < 0 || blk >= rows.num_blocks) {
        if (h == 0) set_error(GPT2_DEVERR_BLOCK);
        blk = 0;
      }
      tbl_s[i] = blk;
    }
  }
  __syncthreads();
  // row index of cache position j of (b, h)
  auto row = [&](int j) -> size_t {
    if (rows.table == nullptr) return (static_cast<size_t>(b) * NH + h) * rows.maxT + j;
    return ((static_cast<size_t>(tbl_s[j >> rows.lbs]) * NH + h) << rows.lbs) + (j & ((1 << rows.lbs) - 1));
  };
  // Cache rows [0, pos) (written by earlier steps) come through a ring of
  // kDecStages chunks in shared memory, copied by the last warp with bulk
  // copies (one per run of consecutive rows: the whole chunk in the dense
  // layout, up to a block boundary in the paged one); the first kDecStages
  // chunks are requested before the wait for the QKV projection, which
  // leaves HBM mostly idle.  (With each warp loading its chunk into
  // registers and waiting for it in turn, the kernel kept one chunk per warp
  // in flight: measured, about 12 us per layer inside a decode step.)
  const int n_cached = pos_ok ? (pos + kChunk - 1) / kChunk : 0;  // chunks with cache rows
  uint32_t filled = 0, fill_par = 0;  // producer: stages ever filled, parity of their last fill
  int issued = 0;
  auto issue = [&](int c) -> bool {  // producer lane: chunk c into stage c % kDecStages
    const int st = c % kDecStages;
    if (c >= kDecStages && !mbar_wait(&empty[st], ((c / kDecStages) - 1) & 1)) return false;
    const int j0 = c * kChunk, j1 = min(j0 + kChunk, pos);
    uint8_t* kdst = dec_smem + st * kDecStageBytes;
    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>((j1 - j0) * kRowBytes * 2));
    for (int j = j0; j < j1;) {
      const int run_end = rows.table == nullptr ? j1 : min(j1, ((j >> rows.lbs) + 1) << rows.lbs);
      const uint32_t bytes = static_cast<uint32_t>((run_end - j) * kRowBytes);
      const size_t rj = row(j) * HS;
      bulk_load(kdst + (j - j0) * kRowBytes, kcache + rj, bytes, &full[st]);
      bulk_load(kdst + kDecStageBytes / 2 + (j - j0) * kRowBytes, vcache + rj, bytes, &full[st]);
      j = run_end;
    }
    filled |= 1u << st;
    fill_par = (fill_par & ~(1u << st)) | ((static_cast<uint32_t>(c / kDecStages) & 1u) << st);
    ++issued;
    return true;
  };
  const bool producer = warp == kDecWarps;
  bool prod_ok = true;
  if (producer && lane == 0)
    for (int c = 0; c < min(n_cached, kDecStages) && prod_ok; ++c) prod_ok = issue(c);
  pdl_wait();  // q and this token's key and value come from the QKV projection
  pdl_trigger();
  float m = -INFINITY, l = 0.f, acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  if (producer) {
    if (lane == 0) {
      for (int c = issued; c < n_cached && prod_ok; ++c) prod_ok = issue(c);
      // the copies issued here land before the CTA may exit
      for (int st = 0; st < kDecStages; ++st)
        if ((filled >> st) & 1u) mbar_wait(&full[st], (fill_par >> st) & 1u);
    }
    __syncwarp();
  } else if (!pos_ok) {  // a position outside the cache: flagged, the row's output is zero
    if (threadIdx.x == 0) set_error(GPT2_DEVERR_POSITION);
    for (int d = threadIdx.x; d < HS; d += 32 * kDecWarps) out[static_cast<size_t>(b) * C + h * HS + d] = from_f32<OutT>(0.f);
  } else {
    // the query's dimensions of this lane, scaled by log2(e) / sqrt(hs)
    float q[kPer];
    {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(b) * 3 * C + h * HS) + dg);
      const E* e = reinterpret_cast<const E*>(&raw);
#pragma unroll
      for (int k = 0; k < kPer; ++k) q[k] = to_f32(e[k]) * scale_log2;
    }
    // this token's key and value: used for position pos, and appended
    const uint4* kq = reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(b) * 3 * C + C + h * HS) + dg;
    const uint4* vq = reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(b) * 3 * C + 2 * C + h * HS) + dg;
    if (threadIdx.x < kLPR) {
      reinterpret_cast<uint4*>(kcache + row(pos) * HS)[dg] = __ldg(kq);
      reinterpret_cast<uint4*>(vcache + row(pos) * HS)[dg] = __ldg(vq);
    }
    const int nchunk = pos / kChunk + 1;  // chunks covering positions 0 .. pos
    // K and V rows of chunk c into registers: rows before pos from the
    // chunk's stage (its copy waited for, the stage freed once read), row pos
    // from the QKV row, zero past pos
    auto load = [&](int c, uint4(&kr)[kIt], uint4(&vr)[kIt]) -> bool {
      const int j0 = c * kChunk;
      const bool staged = c < n_cached;
      const int st = c % kDecStages;
      if (staged && !__all_sync(0xffffffffu, mbar_wait(&full[st], (c / kDecStages) & 1))) return false;
      const uint8_t* kst = dec_smem + st * kDecStageBytes;
#pragma unroll
      for (int i = 0; i < kIt; ++i) {
        const int r = g + i * kRPI, j = j0 + r;
        if (j < pos) {
          kr[i] = reinterpret_cast<const uint4*>(kst + r * kRowBytes)[dg];
          vr[i] = reinterpret_cast<const uint4*>(kst + kDecStageBytes / 2 + r * kRowBytes)[dg];
        } else if (j == pos) {
          kr[i] = __ldg(kq);
          vr[i] = __ldg(vq);
        } else {
          kr[i] = make_uint4(0u, 0u, 0u, 0u);
          vr[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (staged) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      return true;
    };
    // the online softmax over chunk c's rows
    auto consume = [&](int c, const uint4(&kr)[kIt], const uint4(&vr)[kIt]) {
      const int j0 = c * kChunk + g;
      // scores (log2 units) of this lane's kIt rows; the row's kLPR lanes
      // each hold a partial dot product and sum it by shuffles
      float sc[kIt];
      float cmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < kIt; ++i) {
        const E* e = reinterpret_cast<const E*>(&kr[i]);
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < kPer; ++k) d = fmaf(q[k], to_f32(e[k]), d);
#pragma unroll
        for (int o = kLPR / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        sc[i] = (j0 + i * kRPI <= pos) ? d : -INFINITY;
        cmax = fmaxf(cmax, sc[i]);
      }
#pragma unroll
      for (int o = 16; o >= kLPR; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      // position c * kChunk <= pos is in the chunk, so cmax is finite
      const float m_new = fmaxf(m, cmax);
      const float alpha = exp2_approx(m - m_new);  // 0 on the first chunk (m = -inf)
      l *= alpha;
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] *= alpha;
#pragma unroll
      for (int i = 0; i < kIt; ++i) {
        const float p = exp2_approx(sc[i] - m_new);  // 0 past pos
        l += p;
        const E* e = reinterpret_cast<const E*>(&vr[i]);
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc[k] = fmaf(p, to_f32(e[k]), acc[k]);
      }
      m = m_new;
    };
    // this warp's chunks c = warp, warp + kDecWarps, ...
    for (int c = warp; c < nchunk; c += kDecWarps) {
      uint4 kr[kIt], vr[kIt];
      if (!load(c, kr, vr)) break;
      consume(c, kr, vr);
    }
  }
  // sum over the rows of an instruction: every lane then holds the warp's
  // sum and its dimensions' output
#pragma unroll
  for (int o = 16; o >= kLPR; o >>= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
  }
  if (!producer) {
    if (lane == 0) {
      m_s[warp] = m;
      l_s[warp] = l;
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) o_s[warp][dg * kPer + k] = acc[k];
    }
  }
  __syncthreads();
  if (!pos_ok) return;
  for (int d = threadIdx.x; d < HS; d += blockDim.x) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, m_s[w]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      if (m_s[w] == -INFINITY) continue;  // a warp that had no chunk
      const float f = exp2_approx(m_s[w] - M);
      L = fmaf(l_s[w], f, L);
      O = fmaf(o_s[w][d], f, O);
    }
    out[static_cast<size_t>(b) * C + h * HS + d] = from_f32<OutT>(O / L);
  }
}

}  // namespace

template <int HS, typename T16>
static void attention_tc_hs(void* out, bool out16, const void* qkv, int B, int T, int C, int NH, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HS));
  dim3 grid((T + kBQ - 1) / kBQ, NH, B);
  const uint16_t* q = static_cast<const uint16_t*>(qkv);
  if (out16)
    attn_tc_kernel<HS, T16, true><<<grid, kAttnThreads, 0, s>>>(out, q, T, C, scale_log2);
  else
    attn_tc_kernel<HS, T16, false><<<grid, kAttnThreads, 0, s>>>(out, q, T, C, scale_log2);
}

template <typename T16>
static int attention_tc(void* out, bool out16, const void* qkv, int B, int T, int C, int NH, cudaStream_t s) {
  switch (C / NH) {
    case 16: attention_tc_hs<16, T16>(out, out16, qkv, B, T, C, NH, s); return GPT2_OK;
    case 32: attention_tc_hs<32, T16>(out, out16, qkv, B, T, C, NH, s); return GPT2_OK;
  }
  return GPT2_ERR_UNSUPPORTED;
}

int launch_attention_16(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                        cudaStream_t s) {
  if (C / NH == 64) return launch_attention_tc05(out, out16, qkv, op, B, T, C, NH, s);  // tcgen05 kernel
  if (op == kOpF16) return attention_tc<__half>(out, out16, qkv, B, T, C, NH, s);
  return attention_tc<__nv_bfloat16>(out, out16, qkv, B, T, C, NH, s);
}

int launch_attention_f32(float* out, const float* qkv, int B, int T, int C, int NH, cudaStream_t s) {
  const int hs = C / NH;
  const float scale = 1.0f / sqrtf(static_cast<float>(hs));
  dim3 grid((T + 63) / 64, NH, B);
  switch (hs) {
    case 16: attn_f32_kernel<16><<<grid, 64, 0, s>>>(out, qkv, T, C, scale); return GPT2_OK;
    case 32: attn_f32_kernel<32><<<grid, 64, 0, s>>>(out, qkv, T, C, scale); return GPT2_OK;
    case 64: attn_f32_kernel<64><<<grid, 64, 0, s>>>(out, qkv, T, C, scale); return GPT2_OK;
  }
  return GPT2_ERR_UNSUPPORTED;
}

template <typename E, typename OutT, int HS>
static void decode_typed(OutT* out, const E* qkv, E* kc, E* vc, int B, int C, int NH, int pos, const int* pos_arr,
                         const KVRows& rows, cudaStream_t s) {
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HS));
  // the ring of cache chunks is dynamic shared memory beyond the 48 KB a
  // launch gets without asking (set once per instantiation and device)
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices && !attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_attn_kernel<E, OutT, HS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kDecSmem) == cudaSuccess)
      attr_set[dev] = true;
  }
  launch_pdl(decode_attn_kernel<E, OutT, HS>, dim3(NH, B), dim3(32 * (kDecWarps + 1)), kDecSmem, s, out, qkv, kc, vc,
             C, NH, pos, pos_arr, rows, scale_log2);
}

template <typename E>
static void decode_16(void* out, bool out16, const void* qkv, void* kcache, void* vcache, int B, int C, int NH,
                      int pos, const int* pos_arr, const KVRows& rows, cudaStream_t s) {
  const E* q = static_cast<const E*>(qkv);
  E* kc = static_cast<E*>(kcache);
  E* vc = static_cast<E*>(vcache);
  E* o16 = static_cast<E*>(out);
  float* o32 = static_cast<float*>(out);
  switch (C / NH) {
    case 16:
      if (out16) decode_typed<E, E, 16>(o16, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      else decode_typed<E, float, 16>(o32, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      break;
    case 32:
      if (out16) decode_typed<E, E, 32>(o16, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      else decode_typed<E, float, 32>(o32, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      break;
    default:
      if (out16) decode_typed<E, E, 64>(o16, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      else decode_typed<E, float, 64>(o32, q, kc, vc, B, C, NH, pos, pos_arr, rows, s);
      break;
  }
}

void launch_decode_attention_16(void* out, bool out16, const void* qkv, void* kcache, void* vcache, int op, int B,
                                int C, int NH, int pos, const int* pos_arr, const KVRows& rows, cudaStream_t s) {
  if (op == kOpF16)
    decode_16<__half>(out, out16, qkv, kcache, vcache, B, C, NH, pos, pos_arr, rows, s);
  else
    decode_16<__nv_bfloat16>(out, out16, qkv, kcache, vcache, B, C, NH, pos, pos_arr, rows, s);
}

void launch_decode_attention_f32(float* out, const float* qkv, float* kcache, float* vcache, int B, int C, int NH,
                                 int pos, const int* pos_arr, const KVRows& rows, cudaStream_t s) {
  switch (C / NH) {
    case 16: decode_typed<float, float, 16>(out, qkv, kcache, vcache, B, C, NH, pos, pos_arr, rows, s); break;
    case 32: decode_typed<float, float, 32>(out, qkv, kcache, vcache, B, C, NH, pos, pos_arr, rows, s); break;
    default: decode_typed<float, float, 64>(out, qkv, kcache, vcache, B, C, NH, pos, pos_arr, rows, s); break;
  }
}

}  // namespace gpt2
