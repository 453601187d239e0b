// attention_tc.cu -- causal attention of the GPT-2 forward pass on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); the computation follows Algorithm 1: key/value tiles stream
// through shared memory and each query row keeps a running maximum and sum
// while its unnormalised output accumulates, so the T x T score matrix never
// exists.  Key tiles after a query tile are never visited.
//
// Work unit: a CTA (one per SM) holds two adjacent query tiles of 128 rows,
// A = 2i and B = 2i + 1, of one (sequence, head); B needs one key tile more,
// its diagonal.  The score tiles of both form one sequence of steps (A and B
// take turns on each key tile while both have one; B's last tile follows
// alone) that rotates through three S accumulators in TMEM and three P
// buffers in shared memory, so S of step s + 3 is issued as soon as P of
// step s is ready.
//   warp 0      TMA: the CTA's two Q tiles, then K and V tiles (128 keys x
//               64 dimensions each, 128-byte swizzle; one barrier for both)
//               through a ring of three stages, from the fused QKV buffer
//               viewed as [B][T][3C] (rows past T read as zero);
//   warp 1      TMEM (three S: 128 x 128 fp32; O_A, O_B: 128 x 64 fp32) and
//               the MMAs, S = Q K^T (4 instructions of K = 16) and O += P V
//               (8; V an MN-major operand); the warp runs the issuing loop
//               and one elected lane issues.  It waits once per key tile
//               (K and V land together) and frees the stage with one commit
//               after the tile's last P V: measured, each wait and commit
//               of this warp costs a few hundred cycles in a busy SM, and
//               this warp paces the kernel;
//   warps 2-5   softmax of group A, warps 6-9 softmax of group B, one thread
//               per query row.  One pass over the S row from TMEM in chunks
//               of 32 keys (the next chunk's load in flight): p = exp2(s *
//               scale - m) with the running maximum m as it stands (on the
//               first tile, the maximum of its first chunk), rounded to the
//               16-bit type into swizzled shared memory (the A operand of
//               P V), and the running sum.  A score above m + 8 (log2
//               units) sends the tile through two passes instead: the row
//               maximum, the rescale of O in TMEM and of the sum by
//               2^(m - m_new), then the exponentials.  Exact either way: the
//               final division by the sum uses the same m as the
//               numerators.  At the end O / l goes to [B, T, C].
// Every wait is bounded; a timeout sets the device error word and the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kTQ = 128;   // query rows per query tile = TMEM lanes
constexpr int kTK = 128;   // keys per key tile
constexpr int kHS = 64;    // head size
constexpr int kQBytes = kTQ * kHS * 2;        // 16 KB: 128 rows of 128 bytes
constexpr int kPBytes = kTQ * kTK * 2;        // 32 KB: two 64-key swizzle atoms
constexpr int kRing = 3;   // S accumulators in TMEM and P buffers in shared memory
constexpr int kSoftmaxWarps = 4;  // per group and CTA
constexpr int kThreads = 64 + 2 * 32 * kSoftmaxWarps;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S buffer r at 128 r, O of group x at 384 + 64 x
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = kRing * kTK;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Smem {
  static constexpr int kKBytes = kTK * 128;           // 128 keys x 64 dimensions
  static constexpr int kVBytes = kTK * 128;
  static constexpr int kKV = 3;                        // K/V pipeline stages
  static constexpr int q = 0;                          // group A tile, group B tile
  static constexpr int k = q + 2 * kQBytes;            // kKV stages of K
  static constexpr int v = k + kKV * kKBytes;          // kKV stages of V
  static constexpr int p = v + kKV * kVBytes;          // kRing buffers
  static constexpr int bars = p + kRing * kPBytes;
  // q_full; kv_full[kKV], kv_empty[kKV]; s_full[kRing], p_full[kRing],
  // o_done[kRing]; o_final[2]; drain
  static constexpr int n_bars = 1 + 2 * kKV + 3 * kRing + 2 + 1;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(Smem::alloc <= 232448, "shared memory budget");

// The schedule of score tiles.  Group A (x = 0) visits key tiles
// 0 .. n_a - 1 and group B (x = 1) 0 .. n_b - 1 (n_b = 0: no group B, else
// n_b >= n_a); while both have tile j, step 2j + x; then B's remaining
// tiles (or, with no B, all of A's) one step each.
struct Schedule {
  int n_a, n_b, lo, n_steps;
  __device__ Schedule(int na, int nb) : n_a(na), n_b(nb), lo(nb > 0 ? na : 0), n_steps(na + nb) {}
  __device__ int group(int s) const { return s < 2 * lo ? (s & 1) : (n_b > 0 ? 1 : 0); }
  __device__ int tile(int s) const { return s < 2 * lo ? (s >> 1) : s - lo; }
  __device__ int step(int x, int j) const { return j < lo ? 2 * j + x : lo + j; }
  // the step is the last to use its key/value tile
  __device__ bool last_user(int s) const { return s >= 2 * lo || (s & 1); }
};

// 320 threads = 10 warps, one CTA per SM.  Registers are allotted per SM
// sub-partition (16K each, warps placed round-robin), so the sub-partition
// holding three warps caps a thread at 168 registers.
template <typename T16, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_qkv, OutT* __restrict__ out, float* __restrict__ lse,
                     int T, int C, int Tp, float scale_log2) {
  using L = Smem;
  constexpr int kKV = L::kKV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* q_full = bars;                  // both Q tiles landed
  uint64_t* kv_full = bars + 1;             // [kKV] K and V of a key tile landed
  uint64_t* kv_empty = kv_full + kKV;       // [kKV] the MMAs have read them
  // ring slot r serves steps s = r, r + 3, ...: use k of the slot is phase k
  uint64_t* s_full = kv_empty + kKV;        // [kRing] S of step s is in TMEM
  uint64_t* p_full = s_full + kRing;        // [kRing] P of step s written (every softmax warp of the group)
  uint64_t* o_done = p_full + kRing;        // [kRing] P V of step s done
  uint64_t* o_final = o_done + kRing;       // [group] the group's last P V done (one phase)
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // unit u: query tiles 2u and 2u + 1; the longest units first
  const int u = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  auto q_tile = [&](int x) { return 2 * u + x; };
  const int kv_tiles = (T + kTK - 1) / kTK;
  const int n_a = min(2 * u + 1, kv_tiles);
  const int n_b = (2 * u + 1) * kTQ < T ? min(2 * u + 2, kv_tiles) : 0;
  const Schedule sch(n_a, n_b);
  const int n_kv = max(n_a, n_b);
  constexpr uint32_t kFmt = std::is_same<T16, __half>::value ? 0u : 1u;
  constexpr uint32_t kIdescS = make_idesc(kFmt, kTQ, kTK);
  constexpr uint32_t kIdescPV = make_idesc(kFmt, kTQ, kHS) | (1u << 16);  // B (V) MN-major

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1u);
    for (int i = 0; i < kKV; ++i) {
      mbar_init(&kv_full[i], 1u);
      mbar_init(&kv_empty[i], 1u);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&s_full[r], 1u);
      mbar_init(&p_full[r], kSoftmaxWarps);  // the group's softmax warps
      mbar_init(&o_done[r], 1u);
    }
    for (int x = 0; x < 2; ++x) mbar_init(&o_final[x], 1u);
    mbar_init(drain, 1u);
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
  pdl_wait();  // a programmatic dependent launch: the QKV projection has finished
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      uint32_t filled = 0, par = 0;  // per stage: ever filled; parity of the last fill
      mbar_arrive_expect_tx(q_full, 2 * kQBytes);
      tma_load_3d(smem + L::q, &tmap_qkv, q_full, h * kHS, q_tile(0) * kTQ, b);
      tma_load_3d(smem + L::q + kQBytes, &tmap_qkv, q_full, h * kHS, q_tile(1) * kTQ, b);
      for (int j = 0; j < n_kv && !*abort_flag; ++j) {
        const int st = j % kKV;
        const uint32_t ph = (j / kKV) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], L::kKBytes + L::kVBytes);
        tma_load_3d(smem + L::k + st * L::kKBytes, &tmap_qkv, &kv_full[st], C + h * kHS, j * kTK, b);
        tma_load_3d(smem + L::v + st * L::kVBytes, &tmap_qkv, &kv_full[st], 2 * C + h * kHS, j * kTK, b);
        filled |= 1u << st;
        par = (par & ~(1u << st)) | (ph << st);
      }
      // the copies issued here land before the CTA may exit: this thread
      // alone arms the full barriers, so the phase of a stage's last fill
      // completes exactly when its bytes have landed
      for (int st = 0; st < kKV; ++st)
        if ((filled >> st) & 1u) mbar_wait(&kv_full[st], (par >> st) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    // the whole warp runs the loop, one lane issues
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0));
    const uint32_t q_addr = smem_u32(smem + L::q);
    const uint32_t p_addr = smem_u32(smem + L::p);
    // S(s) = Q_x K_j^T into S buffer s % kRing; the first step of each key
    // tile waits for its K and V (P V of a tile always follows its S)
    auto issue_s = [&](int s) -> bool {
      const int x = sch.group(s), j = sch.tile(s);
      if (s == sch.step(0, j))  // the tile's first step
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[j % kKV], (j / kKV) & 1))) return false;
      tc_fence_after();
      const uint64_t qd = smem_desc_sw128(q_addr + x * kQBytes);
      const uint64_t kd = smem_desc_sw128(smem_u32(smem + L::k + (j % kKV) * L::kKBytes));
#pragma unroll
      for (int kk = 0; kk < kHS / 16; ++kk)  // 16 dimensions = 32 bytes = 2 in the descriptor's address field
        tc_mma_warp<false>(tmem + kTmemS + (s % kRing) * kTK, qd + 2 * kk, kd + 2 * kk, kIdescS, kk > 0 ? 1u : 0u);
      tc_commit_warp(&s_full[s % kRing]);
      return true;
    };
    // O_x += P(s) V_j
    auto issue_pv = [&](int s) -> bool {
      const int x = sch.group(s), j = sch.tile(s);
      if (!__all_sync(0xffffffffu, mbar_wait(&p_full[s % kRing], (s / kRing) & 1))) return false;
      tc_fence_after();
      const uint32_t v_addr = smem_u32(smem + L::v + (j % kKV) * L::kVBytes);
      const uint64_t pd = smem_desc_sw128(p_addr + (s % kRing) * kPBytes);
      const uint64_t vd = smem_desc_sw128_mn(v_addr, 1024);
#pragma unroll
      for (int kk = 0; kk < kTK / 16; ++kk)  // P: 16 keys = 32 bytes of a 64-key atom; V: 16 rows of 128 bytes
        tc_mma_warp<false>(tmem + kTmemO + x * kHS, pd + ((kk >> 2) * (kPBytes / 2) + (kk & 3) * 32) / 16,
                           vd + kk * (2048 / 16), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit_warp(&o_done[s % kRing]);
      if (j == (x == 0 ? sch.n_a : sch.n_b) - 1) tc_commit_warp(&o_final[x]);
      if (sch.last_user(s)) tc_commit_warp(&kv_empty[j % kKV]);
      return true;
    };
    // S of the first three steps, then per step: P V, and S of the step
    // three later into the S buffer this step has finished reading
    for (int s = 0; s < kRing && s < sch.n_steps && ok; ++s) ok = issue_s(s);
    for (int s = 0; s < sch.n_steps && ok; ++s) {
      ok = issue_pv(s);
      if (ok && s + kRing < sch.n_steps) ok = issue_s(s + kRing);
    }
    if (!ok && lane == 0) *abort_flag = 1;
    tc_commit_warp(drain);
    mbar_wait(drain, 0);
  } else {
    // ---------------------------------------------------------- softmax
    const int x = (warp - 2) / kSoftmaxWarps;  // group: 0 = A (warps 2-5), 1 = B (warps 6-9)
    const int qw = warp & 3;                   // TMEM lane quadrant this warp may access
    const int row = qw * 32 + lane;            // query row within the tile = TMEM lane
    const int t = q_tile(x) * kTQ + row;       // position in the sequence
    const int n_x = x == 0 ? sch.n_a : sch.n_b;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const int t_end = min(t + 1, T);  // keys < t_end are visible to this row
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_x; ++j) {
      const int s = sch.step(x, j), r = s % kRing;
      const uint32_t s_col = kTmemS + r * kTK;
      uint8_t* pbase = smem + L::p + r * kPBytes + row * 128;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[r], (s / kRing) & 1)))) break;
      tc_fence_after();
      // visible keys of this tile: all 128 or up to the diagonal
      const int valid = max(0, min(t_end - j * kTK, kTK));
      // chunks of 32 keys that some row of this warp sees; the rest of the
      // row's P is zero (the upper triangle of the diagonal tile) and its
      // exponentials are not computed
      const int n_live = (__reduce_max_sync(0xffffffffu, valid) + 31) >> 5;
      const bool all_full = __all_sync(0xffffffffu, valid == kTK);
      // P V of this group's previous step s_prev (tile j - 1) must be done
      // before O is rescaled.  Its ring slot's barrier is unambiguous then:
      // P V of step s_prev - 3 finished before S of step s (issued after
      // it), and P V of step s_prev + 3 > s cannot have been issued, as P V
      // goes in step order and that of step s needs this thread's P.
      const int s_prev = j > 0 ? sch.step(x, j - 1) : 0;
      float2 sum2 = make_float2(0.f, 0.f);
      auto store_p = [&](int c, const uint32_t(&pk)[16]) {
        // 32 keys = 4 chunks of 16 bytes: atom c / 2, chunks (c % 2) * 4 + 0..3
        uint8_t* prow = pbase + (c >> 1) * (kPBytes / 2);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = (c & 1) * 4 + q;
          *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      };
      // x = s * scale - m for the 32 keys of a chunk (-inf for masked
      // keys), then p = exp2(x) on the SFU in fp32, rounded to the 16-bit
      // type into P, and their fp32 sum added to sum2.  The exponentials do
      // not wait for the overflow test: a chunk with a key above m + 8
      // (log2 units; a maximum that must be raised) is computed, found, and
      // neither stored nor summed, and the function returns false.  Four
      // independent chains for the maximum and the sum keep the SFU fed.
      auto softmax_chunk = [&](int c, const uint32_t(&cur)[32], bool check) -> bool {
        const float2 sc = make_float2(scale_log2, scale_log2), nm = make_float2(-m_run, -m_run);
        float2 xv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          xv[i] = __ffma2_rn(make_float2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), sc, nm);
        if (!all_full) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (c * 32 + 2 * i >= valid) xv[i].x = -INFINITY;
            if (c * 32 + 2 * i + 1 >= valid) xv[i].y = -INFINITY;
          }
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float2 sq[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          mq[i & 3] = fmax3(mq[i & 3], xv[i].x, xv[i].y);
          const float2 p = make_float2(ex2(xv[i].x), ex2(xv[i].y));
          sq[i & 3] = __fadd2_rn(sq[i & 3], p);
          pk[i] = pack2<T16>(p.x, p.y);
        }
        if (check &&
            __any_sync(0xffffffffu, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) > kRescaleThreshold))
          return false;
        sum2 = __fadd2_rn(sum2, __fadd2_rn(__fadd2_rn(sq[0], sq[1]), __fadd2_rn(sq[2], sq[3])));
        store_p(c, pk);
        return true;
      };
      auto zero_chunk = [&](int c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
        store_p(c, pk);
      };
      // Single pass over the live chunks with the running maximum as it
      // stands, the next chunk's TMEM load in flight while one is
      // processed.  On the first tile the running maximum starts as the
      // maximum of the first chunk's visible scores.  A score above m + 8
      // (log2 units; a maximum that must be raised) stops it, and the tile
      // is redone in two passes below.
      bool done = false;
      {
        uint32_t ra[32], rb[32];
        bool go = true;
        if (n_live > 0) {
          tmem_ld_32x32b_x32(lane_base + s_col, ra);
          tmem_ld_wait_regs(ra);
          if (j == 0) {  // valid >= 1 on every row here
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (all_full || e < valid) mx = fmaxf(mx, __uint_as_float(ra[e]));
            m_run = mx * scale_log2;
          }
        }
        auto chunk = [&](auto cc, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
          constexpr int c = decltype(cc)::value;
          if (!go) return;
          if (c >= n_live) {
            zero_chunk(c);
            return;
          }
          if (c + 1 < n_live) tmem_ld_32x32b_x32(lane_base + s_col + (c + 1) * 32, nxt);
          go = softmax_chunk(c, cur, true);
          if (c + 1 < n_live) tmem_ld_wait_regs(nxt);
        };
        static_assert(kTK == 128, "four chunks of 32 keys");
        chunk(std::integral_constant<int, 0>(), ra, rb);
        chunk(std::integral_constant<int, 1>(), rb, ra);
        chunk(std::integral_constant<int, 2>(), ra, rb);
        chunk(std::integral_constant<int, 3>(), rb, ra);
        done = go;
      }
      if (!done) {
        // Two passes (a maximum that grows by more than 2^8): the row
        // maximum over the tile, the rescale of O and of the running sum,
        // then the exponentials.
        sum2 = make_float2(0.f, 0.f);
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < kTK / 32; ++c) {  // pass 1: the row maximum
          uint32_t rr[32];
          tmem_ld_32x32b_x32(lane_base + s_col + c * 32, rr);
          tmem_ld_wait_regs(rr);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e < valid) mx = fmaxf(mx, __uint_as_float(rr[e]));
        }
        const float m_new = fmaxf(m_run, mx * scale_log2);  // the scale is positive: it commutes with max
        const bool grow = (m_new - m_run) > kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {
          if (j > 0) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[s_prev % kRing], (s_prev / kRing) & 1))))
              break;
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
        // pass 2: p = exp2(s * scale - m) into P(s) (its buffer is free: P V
        // of step s - 3 finished before S of step s)
#pragma unroll 1
        for (int c = 0; c < kTK / 32; ++c) {
          uint32_t rr[32];
          tmem_ld_32x32b_x32(lane_base + s_col + c * 32, rr);
          tmem_ld_wait_regs(rr);
          softmax_chunk(c, rr, false);
        }
      }
      l_run += sum2.x + sum2.y;
      fence_proxy_async_smem();  // P written by this thread becomes visible to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[r]);
    }
    if (ok && n_x > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_final[x], 0));
    if (ok && n_x > 0) {
      tc_fence_after();
      const float inv = 1.0f / l_run;
      // the row's log-sum-exp in log2 units, m + log2(l), for the backward
      if (lse != nullptr && t < T)
        lse[(static_cast<size_t>(b) * gridDim.y + h) * Tp + t] = m_run + __log2f(l_run);
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
    } else if (!ok) {
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

template <typename T16, typename OutT>
int launch_typed(void* out, float* lse, const CUtensorMap& map, int B, int T, int C, int NH, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};  // per template instance and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  auto kern = attn_tc05_kernel<T16, OutT>;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  const int units = (T + 2 * kTQ - 1) / (2 * kTQ);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units, NH, B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Smem::alloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits for its predecessor itself
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_on() ? 1 : 0;
  const int Tp = (T + kTQ - 1) / kTQ * kTQ;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, static_cast<OutT*>(out), lse, T, C, Tp, scale_log2);
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}
}  // namespace

// qkv [B,T,3C] of the 16-bit operand type op; out [B,T,C] of that type
// (out16) or fp32; lse (optional) [B][NH][Tp], Tp = T rounded up to 128:
// each row's log-sum-exp of the scaled scores in log2 units.  Head size 64
// only.
int launch_attention_tc05(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                          cudaStream_t s, float* lse) {
  if (C / NH != kHS || C % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  // [B][T][3C] viewed as tiles of 64 dimensions x 128 rows with the 128-byte
  // swizzle: Q, K (K-major operands) and V (an MN-major operand) alike
  CUtensorMap map;
  const uint64_t dims[3] = {static_cast<uint64_t>(3 * C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[2] = {static_cast<uint64_t>(3 * C) * 2, static_cast<uint64_t>(T) * 3 * C * 2};
  const uint32_t box[3] = {kHS, kTQ, 1};
  const CUtensorMapDataType dt = op == kOpF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tensor_map(&map, dt, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return GPT2_ERR_CUDA;
  if (op == kOpF16)
    return out16 ? launch_typed<__half, __half>(out, lse, map, B, T, C, NH, s)
                 : launch_typed<__half, float>(out, lse, map, B, T, C, NH, s);
  return out16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(out, lse, map, B, T, C, NH, s)
               : launch_typed<__nv_bfloat16, float>(out, lse, map, B, T, C, NH, s);
}

}  // namespace gpt2
