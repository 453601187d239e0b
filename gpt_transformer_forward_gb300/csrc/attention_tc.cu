// attention_tc.cu -- causal attention of the GPT-2 forward pass on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); the computation follows Algorithm 1: key/value tiles stream
// through shared memory and each query row keeps a running maximum and sum
// while its unnormalised output accumulates, so the T x T score matrix never
// exists.  Key tiles after a query tile are never visited.
//
// Work unit: the one-CTA form (the default) gives a CTA (one per SM) two
// adjacent query tiles of 128 rows, A = 2i and B = 2i + 1, of one (sequence,
// head); B needs one key tile more, its diagonal.  The pair form gives a
// cluster of two CTAs four tiles, 4i .. 4i + 3: CTA r holds tile 4i + r of
// group A and 4i + 2 + r of group B, and each MMA is a paired tcgen05
// instruction (cta_group::2, M = 256) over one group's two tiles, issued by
// the even CTA; each CTA loads half of every K tile (keys 64r .. 64r + 63:
// the B operand of S is split by N = keys) and of every V tile (dimensions
// 32r .. 32r + 31, MN-major with the 64-byte swizzle: P V's B operand is
// split by N = head dimension), and the tile after the diagonal of the even
// CTA's rows is computed for the odd CTA's and fully masked.
//
// The score tiles of both groups form one sequence of steps (A and B take
// turns on each key tile while both have one; B's last tile or tiles follow
// alone) that rotates through three S accumulators in TMEM and three P
// buffers in shared memory, so S of step s + 3 is issued as soon as P of
// step s is ready and a softmax rarely waits for the tensor cores.
//   warp 0      TMA: the CTA's two Q tiles, then its K and V tiles (or
//               halves) through a ring of stages, from the fused QKV buffer
//               viewed as [B][T][3C] (rows past T read as zero);
//   warp 1      TMEM (three S: 128 x 128 fp32; O_A, O_B: 128 x 64 fp32) and
//               the MMAs, S = Q K^T (4 instructions of K = 16) and O += P V
//               (8); the warp runs the issuing loop and one elected lane
//               issues (in a pair, the even CTA's warp for both);
//   warps 2-5   softmax of group A, warps 6-9 softmax of group B, one thread
//               per query row.  On a tile after the first, one pass over
//               the S row from TMEM in chunks of 32 keys (the next chunk's
//               load in flight): p = exp2(s*scale - m) with the running
//               maximum m as it stands, rounded to the 16-bit type into
//               swizzled shared memory (the A operand of P V), running sum.
//               A score above m + 8 (log2 units; always on the first tile)
//               sends the tile through two passes instead: the row maximum,
//               the rescale of O in TMEM and of the sum by 2^(m - m_new),
//               then the exponentials.  Exact either way: the final
//               division by the sum uses the same m as the numerators.  At
//               the end O / l goes to [B, T, C].
// Every wait is bounded; a timeout sets the device error word and the CTA
// (pair) drains its copies and MMAs, frees TMEM and returns.
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

// The pair form (kPair) and the one-CTA form differ in the share of each K
// and V tile a CTA loads and in how many K/V stages fit.
template <bool kPair>
struct Smem {
  static constexpr int kCTAs = kPair ? 2 : 1;
  static constexpr int kKBytes = kTK / kCTAs * 128;  // keys x 64 dims
  static constexpr int kVBytes = kTK * 128 / kCTAs;  // 128 keys x dims
  static constexpr int kKV = kPair ? 4 : 3;          // K and V pipeline stages
  static constexpr int q = 0;                         // group A tile, group B tile
  static constexpr int k = q + 2 * kQBytes;           // kKV stages of K
  static constexpr int v = k + kKV * kKBytes;         // kKV stages of V
  static constexpr int p = v + kKV * kVBytes;         // kRing buffers
  static constexpr int bars = p + kRing * kPBytes;
  // q_full; k_full[kKV], k_empty[kKV], v_full[kKV], v_empty[kKV];
  // s_full[kRing], p_full[kRing], o_done[kRing]; o_final[2]; drain
  static constexpr int n_bars = 1 + 4 * kKV + 3 * kRing + 2 + 1;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(Smem<true>::alloc <= 232448 && Smem<false>::alloc <= 232448, "shared memory budget");

// The pair's schedule of score tiles.  Group A (x = 0) visits key tiles
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
// holding three warps caps a thread at 168 registers; the softmax threads
// therefore read their S row in halves instead of holding all of it.
template <typename T16, typename OutT, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, OutT* __restrict__ out, int T, int C,
                   float scale_log2) {
  using L = Smem<kPair>;
  constexpr int kKV = L::kKV;
  constexpr uint32_t kCTAs = L::kCTAs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* q_full = bars;                  // even CTA: both CTAs' Q tiles landed
  uint64_t* k_full = bars + 1;              // [kKV] even CTA: both K halves landed
  uint64_t* k_empty = k_full + kKV;         // [kKV] both CTAs: the MMAs have read K
  uint64_t* v_full = k_empty + kKV;         // [kKV] even CTA
  uint64_t* v_empty = v_full + kKV;         // [kKV] both CTAs
  // ring slot r serves steps s = r, r + 3, ...: use k of the slot is phase k
  uint64_t* s_full = v_empty + kKV;         // [kRing] both CTAs: S of step s is in TMEM
  uint64_t* p_full = s_full + kRing;        // [kRing] even CTA: P of step s written (every softmax warp)
  uint64_t* o_done = p_full + kRing;        // [kRing] both CTAs: P V of step s done
  uint64_t* o_final = o_done + kRing;       // [group] both CTAs: the group's last P V done (one phase)
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  // unit u: query tiles 4u .. 4u + 3 of a pair, 2u and 2u + 1 of one CTA;
  // the longest units first
  const int u = static_cast<int>(gridDim.x / kCTAs) - 1 - static_cast<int>(blockIdx.x / kCTAs);
  const int h = blockIdx.y, b = blockIdx.z;
  auto q_tile = [&](int x) { return kPair ? 4 * u + 2 * x + static_cast<int>(rank) : 2 * u + x; };
  const int kv_tiles = (T + kTK - 1) / kTK;
  const int last_a = kPair ? 4 * u + 1 : 2 * u;  // the last query tile of each group
  const int n_a = min(last_a + 1, kv_tiles);
  const int n_b = (last_a + 1) * kTQ < T ? min(last_a + kCTAs + 1, kv_tiles) : 0;
  const Schedule sch(n_a, n_b);
  const int n_kv = max(n_a, n_b);
  constexpr uint32_t kFmt = std::is_same<T16, __half>::value ? 0u : 1u;
  constexpr uint32_t kIdescS = make_idesc(kFmt, kCTAs * kTQ, kTK);
  constexpr uint32_t kIdescPV = make_idesc(kFmt, kCTAs * kTQ, kHS) | (1u << 16);  // B (V) MN-major

  if (threadIdx.x == 0) {
    mbar_init(q_full, kCTAs);
    for (int i = 0; i < kKV; ++i) {
      mbar_init(&k_full[i], kCTAs);
      mbar_init(&k_empty[i], 1u);
      mbar_init(&v_full[i], kCTAs);
      mbar_init(&v_empty[i], 1u);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&s_full[r], 1u);
      mbar_init(&p_full[r], kCTAs * kSoftmaxWarps);  // the group's softmax warps (of both CTAs)
      mbar_init(&o_done[r], 1u);
    }
    for (int x = 0; x < 2; ++x) mbar_init(&o_final[x], 1u);
    mbar_init(drain, 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
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
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // a programmatic dependent launch: the QKV projection has finished
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      uint32_t k_filled = 0, v_filled = 0, par = 0;  // per stage: K, V ever filled; parity of the last fill
      // one load into this CTA's shared memory, completing on the even CTA's
      // barrier in a pair
      auto load = [&](void* dst, const CUtensorMap* map, uint64_t* bar, uint32_t bytes, int xc, int yc) {
        if constexpr (kPair) {
          const uint32_t bar0 = mapa_shared(smem_u32(bar), 0);
          mbar_arrive_expect_tx_cluster(bar0, bytes);
          tma_load_3d_pair(dst, map, bar0, xc, yc, b);
        } else {
          mbar_arrive_expect_tx(bar, bytes);
          tma_load_3d(dst, map, bar, xc, yc, b);
        }
      };
      if constexpr (kPair) {
        const uint32_t q_full0 = mapa_shared(smem_u32(q_full), 0);
        mbar_arrive_expect_tx_cluster(q_full0, 2 * kQBytes);
        tma_load_3d_pair(smem + L::q, &tmap_q, q_full0, h * kHS, q_tile(0) * kTQ, b);
        tma_load_3d_pair(smem + L::q + kQBytes, &tmap_q, q_full0, h * kHS, q_tile(1) * kTQ, b);
      } else {
        mbar_arrive_expect_tx(q_full, 2 * kQBytes);
        tma_load_3d(smem + L::q, &tmap_q, q_full, h * kHS, q_tile(0) * kTQ, b);
        tma_load_3d(smem + L::q + kQBytes, &tmap_q, q_full, h * kHS, q_tile(1) * kTQ, b);
      }
      for (int j = 0; j < n_kv && !*abort_flag; ++j) {
        const int st = j % kKV;
        const uint32_t ph = (j / kKV) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        load(smem + L::k + st * L::kKBytes, &tmap_k, &k_full[st], L::kKBytes, C + h * kHS,
             j * kTK + static_cast<int>(rank) * (kTK / 2));
        k_filled |= 1u << st;
        par = (par & ~(1u << st)) | (ph << st);
        if (!mbar_wait(&v_empty[st], ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        load(smem + L::v + st * L::kVBytes, &tmap_v, &v_full[st], L::kVBytes,
             2 * C + h * kHS + static_cast<int>(rank) * (kHS / 2), j * kTK);
        v_filled |= 1u << st;
      }
      // The copies issued here must land before the CTA may exit.  In a pair
      // their completion is counted on the even CTA's barriers, so wait
      // instead for the MMAs that read the last fill of each stage to
      // release it (immediate in the normal case).
      for (int st = 0; st < kKV; ++st) {
        if ((k_filled >> st) & 1u) mbar_wait(&k_empty[st], (par >> st) & 1u);
        if ((v_filled >> st) & 1u) mbar_wait(&v_empty[st], (par >> st) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    if (rank == 0) {  // the whole warp runs the loop, one lane issues
      bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0));
      const uint32_t q_addr = smem_u32(smem + L::q);
      const uint32_t p_addr = smem_u32(smem + L::p);
      auto mma = [&](uint32_t d, uint64_t a, uint64_t bd, uint32_t idesc, uint32_t acc) {
        if constexpr (kPair)
          tc_mma_pair_warp<false>(d, a, bd, idesc, acc);
        else
          tc_mma_warp<false>(d, a, bd, idesc, acc);
      };
      auto commit = [&](uint64_t* bar) {  // in a pair, to the barrier in both CTAs
        if constexpr (kPair)
          tc_commit_pair_warp(bar, 3);
        else
          tc_commit_warp(bar);
      };
      // S(s) = Q_x K_j^T into S buffer s % kRing
      auto issue_s = [&](int s) -> bool {
        const int x = sch.group(s), j = sch.tile(s);
        if (!__all_sync(0xffffffffu, mbar_wait(&k_full[j % kKV], (j / kKV) & 1))) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + L::k + (j % kKV) * L::kKBytes);
#pragma unroll
        for (int kk = 0; kk < kHS / 16; ++kk)
          mma(tmem + kTmemS + (s % kRing) * kTK, smem_desc_sw128(q_addr + x * kQBytes + kk * 32),
              smem_desc_sw128(k_addr + kk * 32), kIdescS, kk > 0 ? 1u : 0u);
        commit(&s_full[s % kRing]);
        if (sch.last_user(s)) commit(&k_empty[j % kKV]);
        return true;
      };
      // O_x += P(s) V_j
      auto issue_pv = [&](int s) -> bool {
        const int x = sch.group(s), j = sch.tile(s);
        // P of both CTAs: written by the softmax threads, released at
        // cluster scope by their arrivals
        if (!__all_sync(0xffffffffu, kPair ? mbar_wait_cluster(&p_full[s % kRing], (s / kRing) & 1)
                                           : mbar_wait(&p_full[s % kRing], (s / kRing) & 1)))
          return false;
        if (!__all_sync(0xffffffffu, mbar_wait(&v_full[j % kKV], (j / kKV) & 1))) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + L::v + (j % kKV) * L::kVBytes);
        const uint32_t pa = p_addr + (s % kRing) * kPBytes;
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          const uint32_t a = pa + (kk >> 2) * (kPBytes / 2) + (kk & 3) * 32;
          // 16 keys = 2 groups of 8 rows of 64 (pair: 32 dims) or 128 bytes
          const uint64_t bv = kPair ? smem_desc_sw64_mn(v_addr + kk * 1024, 512)
                                    : smem_desc_sw128_mn(v_addr + kk * 2048, 1024);
          mma(tmem + kTmemO + x * kHS, smem_desc_sw128(a), bv, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        commit(&o_done[s % kRing]);
        if (j == (x == 0 ? sch.n_a : sch.n_b) - 1) commit(&o_final[x]);
        if (sch.last_user(s)) commit(&v_empty[j % kKV]);
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
      if constexpr (kPair)
        tc_commit_pair_warp(drain, 1);
      else
        tc_commit_warp(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int x = (warp - 2) / kSoftmaxWarps;  // group: 0 = A (warps 2-5), 1 = B (warps 6-9)
    const int qw = warp & 3;                   // TMEM lane quadrant this warp may access
    const int row = qw * 32 + lane;            // query row within the tile = TMEM lane
    const int t = q_tile(x) * kTQ + row;       // position in the sequence
    const int n_x = x == 0 ? sch.n_a : sch.n_b;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const uint32_t p_full0 = kPair ? mapa_shared(smem_u32(p_full), 0) : 0u;
    const int t_end = min(t + 1, T);  // keys < t_end are visible to this row
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_x; ++j) {
      const int s = sch.step(x, j), r = s % kRing;
      const uint32_t s_col = kTmemS + r * kTK;
      uint8_t* pbase = smem + L::p + r * kPBytes + row * 128;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[r], (s / kRing) & 1)))) break;
      tc_fence_after();
      // visible keys of this tile: all 128, up to the diagonal, or none
      // (the tile after the diagonal of the even CTA's rows, computed for
      // the odd CTA's)
      const int valid = max(0, min(t_end - j * kTK, kTK));
      // P V of this group's previous step s_prev (tile j - 1) must be done
      // before O is rescaled.  Its ring slot's barrier is unambiguous then:
      // P V of step s_prev - 3 finished before S of step s (issued after
      // it), and P V of step s_prev + 3 > s cannot have been issued, as P V
      // goes in step order and that of step s needs this thread's P.
      const int s_prev = j > 0 ? sch.step(x, j - 1) : 0;
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      bool done = false;
      if (j > 0) {
        // Single pass: p = exp2(s * scale - m) with the running maximum as
        // it stands, 32 keys at a time, the next chunk's TMEM load in flight
        // while this one is processed.  A score above m + 2^8 (a maximum
        // that must be raised) stops it, and the tile is redone below.
        auto chunk = [&](auto cc, auto masked, uint32_t(&cur)[32], uint32_t(&nxt)[32]) -> bool {
          constexpr int c = decltype(cc)::value;
          constexpr bool kMasked = decltype(masked)::value;
          if (c + 1 < kTK / 32) tmem_ld_32x32b_x32(lane_base + s_col + (c + 1) * 32, nxt);
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float xv = fmaf(__uint_as_float(cur[e]), scale_log2, -m_run);
            if (kMasked && c * 32 + e >= valid) xv = -INFINITY;
            cur[e] = __float_as_uint(xv);
            m4[e & 3] = fmaxf(m4[e & 3], xv);
          }
          const bool over =
              __any_sync(0xffffffffu, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) > kRescaleThreshold);
          if (!over) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0v = ex2(__uint_as_float(cur[e]));  // exp2(-inf) = 0 for masked keys
              const float p1v = ex2(__uint_as_float(cur[e + 1]));
              sum4[(e >> 1) & 3] += p0v + p1v;
              pk[e >> 1] = pack2<T16>(p0v, p1v);
            }
            uint8_t* prow = pbase + (c >> 1) * (kPBytes / 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int ch = (c & 1) * 4 + q;
              *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
          if (c + 1 < kTK / 32) tmem_ld_wait_regs(nxt);
          return !over;
        };
        auto single_pass = [&](auto masked) -> bool {
          uint32_t ra[32], rb[32];
          tmem_ld_32x32b_x32(lane_base + s_col, ra);
          tmem_ld_wait_regs(ra);
          return chunk(std::integral_constant<int, 0>(), masked, ra, rb) &&
                 chunk(std::integral_constant<int, 1>(), masked, rb, ra) &&
                 chunk(std::integral_constant<int, 2>(), masked, ra, rb) &&
                 chunk(std::integral_constant<int, 3>(), masked, rb, ra);
        };
        static_assert(kTK == 128, "four chunks of 32 keys");
        done = __all_sync(0xffffffffu, valid == kTK) ? single_pass(std::false_type())
                                                     : single_pass(std::true_type());
      }
      if (!done) {
        // Two passes (the first tile, or a maximum that grows by more than
        // 2^8): the row maximum, then the exponentials.
        sum4[0] = sum4[1] = sum4[2] = sum4[3] = 0.f;
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {  // pass 1: the row maximum
          uint32_t rr[64];
          tmem_ld_32x32b_x32(lane_base + s_col + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
          tmem_ld_32x32b_x32(lane_base + s_col + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[32]));
          tmem_ld_wait();
          if (valid == kTK) {
#pragma unroll
            for (int e = 0; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(rr[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (half * 64 + e < valid) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(rr[e]));
          }
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m_run, mx * scale_log2);  // the scale is positive: it commutes with max
        const bool grow = (m_new - m_run) > kRescaleThreshold;  // true on the first tile
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
        // pass 2: p = exp2(s * scale - m), rounded to the 16-bit type, into P(s)
        // (its buffer is free: P V of step s - 3 finished before S of step s)
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t rr[64];
          tmem_ld_32x32b_x32(lane_base + s_col + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
          tmem_ld_32x32b_x32(lane_base + s_col + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[32]));
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = half * 2 + c2;  // 32-key chunk of the tile
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int k = c * 32 + e;
              float p0v = ex2(fmaf(__uint_as_float(rr[c2 * 32 + e]), scale_log2, -m_run));
              float p1v = ex2(fmaf(__uint_as_float(rr[c2 * 32 + e + 1]), scale_log2, -m_run));
              if (valid != kTK) {
                if (k >= valid) p0v = 0.f;
                if (k + 1 >= valid) p1v = 0.f;
              }
              sum4[(e >> 1) & 3] += p0v + p1v;
              pk[e >> 1] = pack2<T16>(p0v, p1v);
            }
            // 32 keys = 4 chunks of 16 bytes: atom c / 2, chunks (c % 2) * 4 + 0..3
            uint8_t* prow = pbase + (c >> 1) * (kPBytes / 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int chunk = (c & 1) * 4 + q;
              *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
      }
      l_run += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      fence_proxy_async_smem();  // P written by this thread becomes visible to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_release_cluster(p_full0 + static_cast<uint32_t>(r) * 8u);
        else
          mbar_arrive(&p_full[r]);
      }
    }
    if (ok && n_x > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_final[x], 0));
    if (ok && n_x > 0) {
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
    } else if (!ok) {
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();  // neither CTA leaves while the pair MMAs may read its shared memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

// The one-CTA form is the default: the softmax, not the tensor cores, sets
// the pace of both forms, and the pair form also computes each pair's
// masked tile and couples two CTAs' progress (measured at B = 16, T = 1024:
// 79 us against 97 us per layer).  GPT2_ATTN_PAIR=1 selects the pair form.
bool attention_pair_form() {
  static const int v = [] {
    const char* e = getenv("GPT2_ATTN_PAIR");
    return e ? atoi(e) : 0;
  }();
  return v != 0;
}

template <typename T16, typename OutT, bool kPair>
int launch_typed(void* out, const CUtensorMap* maps, int B, int T, int C, int NH, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};  // per template instance and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(attn_tc05_kernel<T16, OutT, kPair>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<kPair>::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  const int rows_per_unit = (kPair ? 4 : 2) * kTQ;
  const int units = (T + rows_per_unit - 1) / rows_per_unit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((kPair ? 2 : 1) * units, NH, B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Smem<kPair>::alloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  if (kPair) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (pdl_on()) {  // the kernel waits for its predecessor itself
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  // the one-CTA form loads whole K and V tiles: 64 dims x 128 rows, as Q
  const CUtensorMap& mk = kPair ? maps[1] : maps[0];
  const CUtensorMap& mv = kPair ? maps[2] : maps[0];
  auto kern = attn_tc05_kernel<T16, OutT, kPair>;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, maps[0], mk, mv, static_cast<OutT*>(out), T, C, scale_log2);
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}

template <typename T16, typename OutT>
int launch_form(void* out, const CUtensorMap* maps, int B, int T, int C, int NH, cudaStream_t s) {
  return attention_pair_form() ? launch_typed<T16, OutT, true>(out, maps, B, T, C, NH, s)
                               : launch_typed<T16, OutT, false>(out, maps, B, T, C, NH, s);
}
}  // namespace

// qkv [B,T,3C] of the 16-bit operand type op; out [B,T,C] of that type
// (out16) or fp32.  Head size 64 only.
int launch_attention_tc05(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                          cudaStream_t s) {
  if (C / NH != kHS || C % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  // [B][T][3C] viewed three ways: Q tiles (64 dims x 128 rows) and K halves
  // (64 dims x 64 keys), both with the 128-byte swizzle, and V halves
  // (32 dims x 128 keys) with the 64-byte swizzle
  CUtensorMap maps[3];
  const uint64_t dims[3] = {static_cast<uint64_t>(3 * C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t strides[2] = {static_cast<uint64_t>(3 * C) * 2, static_cast<uint64_t>(T) * 3 * C * 2};
  const uint32_t box_q[3] = {kHS, kTQ, 1};
  const uint32_t box_k[3] = {kHS, kTK / 2, 1};
  const uint32_t box_v[3] = {kHS / 2, kTK, 1};
  const CUtensorMapDataType dt = op == kOpF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tensor_map(&maps[0], dt, 3, qkv, dims, strides, box_q, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&maps[1], dt, 3, qkv, dims, strides, box_k, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&maps[2], dt, 3, qkv, dims, strides, box_v, CU_TENSOR_MAP_SWIZZLE_64B))
    return GPT2_ERR_CUDA;
  if (op == kOpF16)
    return out16 ? launch_form<__half, __half>(out, maps, B, T, C, NH, s)
                 : launch_form<__half, float>(out, maps, B, T, C, NH, s);
  return out16 ? launch_form<__nv_bfloat16, __nv_bfloat16>(out, maps, B, T, C, NH, s)
               : launch_form<__nv_bfloat16, float>(out, maps, B, T, C, NH, s);
}

}  // namespace gpt2
