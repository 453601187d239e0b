// attention_tc.cu -- causal attention of the GPT-2 forward pass on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64.
//
// The result is FlashAttention's Algorithm 0 (scores, causal mask, softmax,
// times V); the computation follows Algorithm 1: key/value tiles stream
// through shared memory and each query row keeps a running maximum and sum
// while its unnormalised output accumulates, so the T x T score matrix never
// exists.  Key tiles after a query tile are never visited.
//
// Work unit: two adjacent query tiles of 128 rows, A = 2i and B = 2i + 1, of
// one (sequence, head); B needs one key tile more, its diagonal.  The kernel
// is persistent: one CTA per SM walks a list of units (balanced by length),
// the Q tiles of the next unit load into a second buffer while the current
// one runs, and its steps continue the same rings, so the first loads and
// the epilogue of a unit overlap the work of its neighbours (measured: a
// CTA per unit spent about 5700 cycles before its first S and 1800 in its
// last epilogue, a quarter of the longest unit's time).  The score tiles of
// both form one sequence of steps (A and B take turns on each key tile while
// both have one; B's last tile follows alone) that rotates through three S
// accumulators in TMEM; P of a step is written over the first half of its S
// buffer (16-bit, two per column) and read from there by the P V
// instruction, so S of step s + 3 is issued into that buffer right after P V
// of step s.  S is signalled to each group on a barrier of its own per
// buffer: a group walks only its own steps.
//   warp 0      TMA: per unit its two Q tiles (two buffers), then K and V
//               tiles (128 keys x 64 dimensions each, 128-byte swizzle; one
//               barrier for both) through a ring of three stages, from the
//               fused QKV buffer viewed as [B][T][3C] (rows past T read as
//               zero);
//   warp 1      TMEM (three S: 128 x 128 fp32; O_A, O_B: 128 x 64 fp32) and
//               the S products, S = Q K^T (4 instructions of K = 16), into
//               the ring slot once the P V product three steps back has read
//               it;
//   warp 10     the P V products, O += P V (8 instructions; P the A operand
//               in TMEM, V an MN-major operand in shared memory, so that they
//               read 2 KB of shared memory each instead of 6 KB).  Two
//               issuing warps, not one: measured, a single warp spent about
//               1800 cycles per step issuing 12 instructions and waiting on
//               barriers, three times the tensor work.  Each runs its loop as
//               a whole warp and one elected lane issues.  It waits once per
//               key tile (K and V land together) and frees the stage with
//               one commit after the tile's last P V: measured, each wait
//               and commit of this warp costs a few hundred cycles in a busy
//               SM;
//   warps 2-5   softmax of group A, warps 6-9 softmax of group B, one thread
//               per query row.  One pass over the S row from TMEM in chunks
//               of 32 keys (the next chunk's load in flight): p = exp2(s *
//               scale - m) with the running maximum m as it stands (on the
//               first tile, the maximum of its first chunk), rounded to the
//               16-bit type into TMEM over the chunk's S columns already read
//               (the A operand of P V), and the running sum.  A chunk c whose
//               exponentials sum above 2^8 in a row (as any score above m + 8,
//               log2 units, makes them) stops the pass: the maximum of
//               chunks c.. (those before it are below m + 8), the rescale of
//               O in TMEM, of the sum and of the P chunks already written by
//               2^(m - m_new) where it grows by more than 8 (values that
//               shrink by more than 2^8, so their second rounding is
//               negligible), then the exponentials of
//               chunks c...  Exact either way: the final division by the sum
//               uses the same m as the numerators.  A unit's output is
//               written after the group's first step of its next unit (or at
//               the end), when the unit's last P V has finished: each warp
//               stages its 32 rows of O / l in shared memory and writes them
//               to [B, T, C] with one TMA store (rows past T are clipped):
//               a thread storing its own row to global memory made every
//               16-byte store a separate transaction, and the epilogue took
//               longer than a key tile (measured).
// Every O accumulator is read out (freeing it for the group's next unit)
// before the staged rows are stored.
// Every wait is bounded; a timeout sets the device error word and the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

#include <functional>
#include <queue>
#include <utility>
#include <vector>

namespace gpt2 {
namespace {

constexpr int kTQ = 128;   // query rows per query tile = TMEM lanes
constexpr int kTK = 128;   // keys per key tile
constexpr int kHS = 64;    // head size
constexpr int kQBytes = kTQ * kHS * 2;        // 16 KB: 128 rows of 128 bytes
constexpr int kRing = 3;   // S accumulators (and P) in TMEM
constexpr int kSoftmaxWarps = 4;  // per group and CTA
constexpr int kPvWarp = 2 + 2 * kSoftmaxWarps;  // the warp issuing the P V products
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S buffer r at 128 r, O of group x at 384 + 64 x
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = kRing * kTK;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kRescaleSum = 256.0f;      // 2^kRescaleThreshold

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Smem {
  static constexpr int kKBytes = kTK * 128;           // 128 keys x 64 dimensions
  static constexpr int kVBytes = kTK * 128;
  static constexpr int kKV = 3;                        // K/V pipeline stages
  static constexpr int q = 0;                          // two buffers of (group A tile, group B tile)
  static constexpr int k = q + 4 * kQBytes;            // kKV stages of K
  static constexpr int v = k + kKV * kKBytes;          // kKV stages of V
  static constexpr int stage = v + kKV * kVBytes;      // output staging: 32 rows x 64 fp32 per softmax warp
  static constexpr int kStageBytes = 32 * kHS * 4;
  static constexpr int bars = stage + 2 * kSoftmaxWarps * kStageBytes;
  // q_full[2], q_empty[2]; kv_full[kKV], kv_empty[kKV]; s_full[2][kRing],
  // p_full[kRing], o_done[kRing]; o_final[2], o_free[2]; drain
  static constexpr int n_bars = 4 + 2 * kKV + 4 * kRing + 4 + 1;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(Smem::alloc <= 232448, "shared memory budget");

// The schedule of score tiles of a unit.  Group A (x = 0) visits key tiles
// 0 .. n_a - 1 and group B (x = 1) 0 .. n_b - 1 (n_b = 0: no group B, else
// n_b >= n_a); while both have tile j, step 2j + x; then B's remaining
// tiles (or, with no B, all of A's) one step each.
struct Schedule {
  int n_a, n_b, lo, n_steps;
  __device__ Schedule() : n_a(0), n_b(0), lo(0), n_steps(0) {}
  __device__ Schedule(int na, int nb) : n_a(na), n_b(nb), lo(nb > 0 ? na : 0), n_steps(na + nb) {}
  __device__ int group(int s) const { return s < 2 * lo ? (s & 1) : (n_b > 0 ? 1 : 0); }
  __device__ int tile(int s) const { return s < 2 * lo ? (s >> 1) : s - lo; }
  __device__ int step(int x, int j) const { return j < lo ? 2 * j + x : lo + j; }
  // the step is the last to use its key/value tile
  __device__ bool last_user(int s) const { return s >= 2 * lo || (s & 1); }
};

// A unit: query tiles 2u and 2u + 1 of one (sequence b, head h).  Units are
// numbered by decreasing length (u from the last), then b, then h.  Which
// CTA takes which units comes from a table made on the host: longest
// first, each unit to the CTA with the least work so far (for B = 16, T =
// 1024, 12 heads on 152 CTAs the busiest CTA has 47 steps, against 50 with
// the rule below; measured, the launch about 1 % shorter).  Past the
// table's size CTA c of G takes units c, 2G - 1 - c, 2G + c, 4G - 1 - c,
// ... (alternate rounds run backwards).
constexpr int kSchedMaxCtas = 160;
constexpr int kSchedMaxUnits = 1600;
struct UnitSchedule {
  int n;                                 // units in the table; 0: no table
  uint16_t first[kSchedMaxCtas + 1];     // CTA c's units are unit[first[c] .. first[c + 1])
  uint16_t unit[kSchedMaxUnits];         // unit numbers, each CTA's in increasing order
};
// a kernel's parameters are at most 4 KB: the table beside two tensor maps
static_assert(sizeof(UnitSchedule) <= 3584, "kernel parameter space");
struct Unit {
  int b, h, u, n_kv;
  Schedule sch;
};
struct UnitList {
  int c, G, n_units, per_u, NH, T, U;
  const UnitSchedule* tab;
  __device__ int id(int i) const {  // the CTA's i-th unit, or -1
    if (tab->n > 0) {
      const int e = tab->first[c] + i;
      return e < tab->first[c + 1] ? static_cast<int>(tab->unit[e]) : -1;
    }
    const int k = i * G + ((i & 1) ? G - 1 - c : c);
    return k < n_units ? k : -1;
  }
  __device__ Unit get(int k) const {
    Unit w;
    w.u = U - 1 - k / per_u;
    const int r = k % per_u;
    w.b = r / NH;
    w.h = r % NH;
    const int kv_tiles = (T + kTK - 1) / kTK;
    const int n_a = min(2 * w.u + 1, kv_tiles);
    const int n_b = (2 * w.u + 1) * kTQ < T ? min(2 * w.u + 2, kv_tiles) : 0;
    w.sch = Schedule(n_a, n_b);
    w.n_kv = max(n_a, n_b);
    return w;
  }
};

// A position in a CTA's sequence of steps over its units: unit i (list
// index), its local step s, and the counts before the unit of global steps
// (g0), key/value tiles (kv0) and units with a group B (n_b_before).
struct Cursor {
  const UnitList* ul;
  int i, k, s, g0, kv0, n_b_before;
  Unit w;
  __device__ explicit Cursor(const UnitList* l) : ul(l), i(0), s(0), g0(0), kv0(0), n_b_before(0) {
    k = ul->id(0);
    if (k >= 0) w = ul->get(k);
  }
  __device__ bool valid() const { return k >= 0; }
  __device__ void advance() {
    if (++s < w.sch.n_steps) return;
    g0 += w.sch.n_steps;
    kv0 += w.n_kv;
    if (w.sch.n_b > 0) ++n_b_before;
    s = 0;
    k = ul->id(++i);
    if (k >= 0) w = ul->get(k);
  }
};

// 352 threads = 11 warps, one CTA per SM, persistent over its units.
// Registers are allotted per SM sub-partition (16K each, warps placed
// round-robin), so a sub-partition holding three warps caps a thread at 168
// registers.
template <typename T16, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_qkv, const __grid_constant__ CUtensorMap tmap_out,
                     float* __restrict__ lse, int B, int T, int NH, int Tp, float scale_log2,
                     const __grid_constant__ UnitSchedule sched) {
  using L = Smem;
  constexpr int kKV = L::kKV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* q_full = bars;                  // [2] both Q tiles of a unit landed (buffer = unit index % 2)
  uint64_t* q_empty = q_full + 2;           // [2] the unit's S products have read them
  uint64_t* kv_full = q_empty + 2;          // [kKV] K and V of a key tile landed
  uint64_t* kv_empty = kv_full + kKV;       // [kKV] the MMAs have read them
  // ring slot r serves global steps g = r, r + 3, ...: use k of the slot is
  // phase k of p_full[r] and o_done[r], whose waiters (the issuing warps)
  // walk every step.  S is signalled per group and slot instead: a group
  // walks only its own steps, and after a unit without steps of its own
  // (a last unit with one query tile) it would be two or more phases of a
  // shared barrier behind, where the parity of the phase it waits for has
  // completed already (that let group B read a slot holding group A's S,
  // measured as wrong rows and a timeout).  Phase k of s_full[x][r] is
  // group x's k-th step in slot r; the S products of its next step there
  // wait for P V of a step that needs this group's P of the one before, so
  // no phase completes before the group has waited for the previous one.
  uint64_t* s_full = kv_empty + kKV;        // [2][kRing] S of step g (of group x) is in TMEM
  uint64_t* p_full = s_full + 2 * kRing;    // [kRing] P of step g written (every softmax warp of the group)
  uint64_t* o_done = p_full + kRing;        // [kRing] P V of step g done
  uint64_t* o_final = o_done + kRing;       // [group] the group's last P V of a unit done
  uint64_t* o_free = o_final + 2;           // [group] the group's epilogue has read O
  uint64_t* drain = o_free + 2;             // both issuing warps' MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = NH * kHS;
  const int U = (T + 2 * kTQ - 1) / (2 * kTQ);  // units per (sequence, head)
  UnitList ul;
  ul.c = blockIdx.x;
  ul.G = gridDim.x;
  ul.per_u = B * NH;
  ul.n_units = U * ul.per_u;
  ul.NH = NH;
  ul.T = T;
  ul.U = U;
  ul.tab = &sched;
  constexpr uint32_t kFmt = std::is_same<T16, __half>::value ? 0u : 1u;
  constexpr uint32_t kIdescS = make_idesc(kFmt, kTQ, kTK);
  constexpr uint32_t kIdescPV = make_idesc(kFmt, kTQ, kHS) | (1u << 16);  // B (V) MN-major

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1u);
      mbar_init(&q_empty[i], 1u);
    }
    for (int i = 0; i < kKV; ++i) {
      mbar_init(&kv_full[i], 1u);
      mbar_init(&kv_empty[i], 1u);
    }
    for (int r = 0; r < 2 * kRing; ++r) mbar_init(&s_full[r], 1u);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&p_full[r], kSoftmaxWarps);  // the group's softmax warps
      mbar_init(&o_done[r], 1u);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&o_final[x], 1u);
      mbar_init(&o_free[x], kSoftmaxWarps);
    }
    mbar_init(drain, 2u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_qkv);
    tma_prefetch_desc(&tmap_out);
  }
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
      uint32_t filled = 0, par = 0;    // per K/V stage: ever filled; parity of the last fill
      uint32_t qfilled = 0, qpar = 0;  // the same per Q buffer
      int f = 0;                       // key/value tiles loaded so far
      for (int i = 0;; ++i) {
        const int k = ul.id(i);
        if (k < 0 || *abort_flag) break;
        const Unit w = ul.get(k);
        const int qb = i & 1;
        const uint32_t qph = (i >> 1) & 1;
        if (!mbar_wait(&q_empty[qb], qph ^ 1)) {  // unit i - 2's S products are done with the buffer
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&q_full[qb], 2 * kQBytes);
        uint8_t* qdst = smem + L::q + qb * 2 * kQBytes;
        tma_load_3d(qdst, &tmap_qkv, &q_full[qb], w.h * kHS, (2 * w.u) * kTQ, w.b);
        tma_load_3d(qdst + kQBytes, &tmap_qkv, &q_full[qb], w.h * kHS, (2 * w.u + 1) * kTQ, w.b);
        qfilled |= 1u << qb;
        qpar = (qpar & ~(1u << qb)) | (qph << qb);
        bool ok = true;
        for (int j = 0; j < w.n_kv; ++j, ++f) {
          const int st = f % kKV;
          const uint32_t ph = (f / kKV) & 1;
          if (!mbar_wait(&kv_empty[st], ph ^ 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[st], L::kKBytes + L::kVBytes);
          tma_load_3d(smem + L::k + st * L::kKBytes, &tmap_qkv, &kv_full[st], C + w.h * kHS, j * kTK, w.b);
          tma_load_3d(smem + L::v + st * L::kVBytes, &tmap_qkv, &kv_full[st], 2 * C + w.h * kHS, j * kTK, w.b);
          filled |= 1u << st;
          par = (par & ~(1u << st)) | (ph << st);
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
      // the copies issued here land before the CTA may exit: this thread
      // alone arms the full barriers, so the phase of a buffer's last fill
      // completes exactly when its bytes have landed
      for (int st = 0; st < kKV; ++st)
        if ((filled >> st) & 1u) mbar_wait(&kv_full[st], (par >> st) & 1u);
      for (int qb = 0; qb < 2; ++qb)
        if ((qfilled >> qb) & 1u) mbar_wait(&q_full[qb], (qpar >> qb) & 1u);
    }
  } else if (warp == 1 || warp == kPvWarp) {
    // ------------------------------------------------------------- MMAs
    // the whole warp runs the loop, one lane issues; each warp walks the
    // CTA's steps with its own cursor.
    // S(g) = Q_x K_j^T into S buffer g % kRing.  The unit's first step waits
    // for its Q tiles, the first step of each key tile for its K and V (P V
    // of a tile always follows its S); the unit's last S frees its Q buffer.
    auto issue_s = [&](const Cursor& cs) -> bool {
      const Schedule& sch = cs.w.sch;
      const int s = cs.s, g = cs.g0 + s, x = sch.group(s), j = sch.tile(s), f = cs.kv0 + j;
      const int qb = cs.i & 1;
      if (s == 0 && !__all_sync(0xffffffffu, mbar_wait(&q_full[qb], (cs.i >> 1) & 1))) return false;
      if (s == sch.step(0, j))  // the tile's first step
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[f % kKV], (f / kKV) & 1))) return false;
      tc_fence_after();
      const uint64_t qd = smem_desc_sw128(smem_u32(smem + L::q + qb * 2 * kQBytes + x * kQBytes));
      const uint64_t kd = smem_desc_sw128(smem_u32(smem + L::k + (f % kKV) * L::kKBytes));
#pragma unroll
      for (int kk = 0; kk < kHS / 16; ++kk)  // 16 dimensions = 32 bytes = 2 in the descriptor's address field
        tc_mma_warp<false>(tmem + kTmemS + (g % kRing) * kTK, qd + 2 * kk, kd + 2 * kk, kIdescS, kk > 0 ? 1u : 0u);
      tc_commit_warp(&s_full[x * kRing + g % kRing]);
      if (s == sch.n_steps - 1) tc_commit_warp(&q_empty[qb]);
      return true;
    };
    // O_x += P(g) V_j.  The group's first tile of a unit overwrites O_x:
    // the group's epilogue of its previous unit must have read it.
    auto issue_pv = [&](const Cursor& cp) -> bool {
      const Schedule& sch = cp.w.sch;
      const int s = cp.s, g = cp.g0 + s, x = sch.group(s), j = sch.tile(s), f = cp.kv0 + j;
      if (!__all_sync(0xffffffffu, mbar_wait(&p_full[g % kRing], (g / kRing) & 1))) return false;
      if (j == 0) {
        const int before = x == 0 ? cp.i : cp.n_b_before;  // the group's earlier units
        if (before > 0 && !__all_sync(0xffffffffu, mbar_wait(&o_free[x], (before - 1) & 1))) return false;
      }
      tc_fence_after();
      const uint32_t v_addr = smem_u32(smem + L::v + (f % kKV) * L::kVBytes);
      const uint32_t p_tmem = tmem + kTmemS + (g % kRing) * kTK;  // P(g): the first 64 columns of S(g)'s buffer
      const uint64_t vd = smem_desc_sw128_mn(v_addr, 1024);
#pragma unroll
      for (int kk = 0; kk < kTK / 16; ++kk)  // P: 16 keys = 8 TMEM columns; V: 16 rows of 128 bytes
        tc_mma_ts_warp(tmem + kTmemO + x * kHS, p_tmem + kk * 8, vd + kk * (2048 / 16), kIdescPV,
                       (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit_warp(&o_done[g % kRing]);
      if (j == (x == 0 ? sch.n_a : sch.n_b) - 1) tc_commit_warp(&o_final[x]);
      if (sch.last_user(s)) tc_commit_warp(&kv_empty[f % kKV]);
      return true;
    };
    bool ok = true;
    if (warp == 1) {
      // S(g) into ring slot g % 3 once P V(g - 3) has read P from it
      for (Cursor cs(&ul); cs.valid() && ok; cs.advance()) {
        const int g = cs.g0 + cs.s;
        if (g >= kRing && !(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[g % kRing], ((g - kRing) / kRing) & 1))))
          break;
        ok = issue_s(cs);
      }
    } else {
      for (Cursor cp(&ul); cp.valid() && ok; cp.advance()) ok = issue_pv(cp);
    }
    if (!ok && lane == 0) *abort_flag = 1;
    tc_commit_warp(drain);
    mbar_wait(drain, 0);
  } else {
    // ---------------------------------------------------------- softmax (warps 2-9)
    const int x = (warp - 2) / kSoftmaxWarps;  // group: 0 = A (warps 2-5), 1 = B (warps 6-9)
    const int qw = warp & 3;                   // TMEM lane quadrant this warp may access
    const int row = qw * 32 + lane;            // query row within the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    bool ok = true;
    int g0 = 0, before = 0;  // global steps and this group's units before the current unit
    uint32_t s_par = 0;      // bit r: parity of this group's next phase of s_full[x][r]
    // A unit's output is written after this group's first step of its next
    // unit (or at the end): by then the unit's last P V has long finished,
    // where waiting for it right after the last step held the group up about
    // 1700 cycles per unit (measured).  O is released as soon as it has been
    // read (the next unit's first P V, which overwrites it, waits for that);
    // O / l goes through the warp's staging rows to [B, T, C] with TMA
    // stores.
    struct Done {
      int k;       // the unit (its number in the unit list), or -1: none pending
      float m, l;  // its rows' final maximum and sum
    };
    Done pend{-1, 0.f, 0.f};
    // `before` counts this group's units up to and including the pending
    // one, whose o_final phase is therefore (before - 1) mod 2
    auto epilogue = [&](Done& dn) -> bool {
      const Unit d = ul.get(dn.k);
      dn.k = -1;
      if (!__all_sync(0xffffffffu, mbar_wait(&o_final[x], (before - 1) & 1))) return false;
      tc_fence_after();
      const int t = (2 * d.u + x) * kTQ + row;
      const float inv = 1.0f / dn.l;
      // the row's log-sum-exp in log2 units, m + log2(l), for the backward
      if (lse != nullptr && t < T) lse[(static_cast<size_t>(d.b) * NH + d.h) * Tp + t] = dn.m + __log2f(dn.l);
      if (lane == 0) bulk_wait_group_read<0>();  // the previous unit's store has read the staging rows
      __syncwarp();
      // boxes of 32 rows x 128 bytes (64 16-bit or 32 fp32 columns) in the
      // 128-byte swizzle the TMA store undoes (16-byte piece q of row r at
      // position q ^ (r mod 8): the warp's stores spread over the banks)
      constexpr int kBoxCols = 128 / static_cast<int>(sizeof(OutT));
      constexpr int kBoxes = kHS / kBoxCols;
      uint8_t* stg = smem + L::stage + (warp - 2) * L::kStageBytes;
      auto stage = [&](int c, const uint32_t(&o)[32]) {  // columns 32 c .. 32 c + 31
        if constexpr (std::is_same<OutT, float>::value) {  // one box row, 8 pieces
          uint8_t* srow = stg + c * 4096 + lane * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(srow + ((q ^ (lane & 7)) << 4)) =
                make_uint4(__float_as_uint(__uint_as_float(o[4 * q + 0]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv));
        } else {  // half a box row, pieces 4c .. 4c + 3
          uint8_t* srow = stg + lane * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack2<T16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            v.y = pack2<T16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            v.z = pack2<T16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            v.w = pack2<T16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            *reinterpret_cast<uint4*>(srow + (((4 * c + q) ^ (lane & 7)) << 4)) = v;
          }
        }
      };
      {
        uint32_t o[32];
        tmem_ld_32x32b_x32(lane_base + kTmemO + x * kHS, o);
        tmem_ld_wait_regs(o);
        stage(0, o);
        tmem_ld_32x32b_x32(lane_base + kTmemO + x * kHS + 32, o);
        tmem_ld_wait_regs(o);
        // O has been read: the next unit's P V may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[x]);
        stage(1, o);
      }
      fence_proxy_async_smem();  // the staged rows become visible to the TMA store
      __syncwarp();
      const int row0 = (2 * d.u + x) * kTQ + qw * 32;  // the warp's first row; rows past T are clipped
      if (lane == 0 && row0 < T) {
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_store_3d(&tmap_out, stg + bx * 4096, d.h * kHS + bx * kBoxCols, row0, d.b);
        bulk_commit_group();
      }
      return true;
    };
    for (int i = 0; ok; ++i) {
      const int k = ul.id(i);
      if (k < 0) break;
      const Unit w = ul.get(k);
      const Schedule& sch = w.sch;
      const int n_x = x == 0 ? sch.n_a : sch.n_b;
      const int b = w.b, h = w.h;
      const int t = (2 * w.u + x) * kTQ + row;  // position in the sequence
      const int t_end = min(t + 1, T);          // keys < t_end are visible to this row
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_x; ++j) {
        const int s = g0 + sch.step(x, j), r = s % kRing;  // the global step
        const uint32_t s_col = kTmemS + r * kTK;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x * kRing + r], (s_par >> r) & 1u)))) break;
        s_par ^= 1u << r;
        tc_fence_after();
        // visible keys of this tile: all 128 or up to the diagonal
        const int valid = max(0, min(t_end - j * kTK, kTK));
        // chunks of 32 keys that some row of this warp sees; the rest of the
        // row's P is zero (the upper triangle of the diagonal tile) and its
        // exponentials are not computed
        const int n_live = (__reduce_max_sync(0xffffffffu, valid) + 31) >> 5;
        const bool all_full = __all_sync(0xffffffffu, valid == kTK);
        // keys below min_valid are visible to every row of the warp: a chunk
        // below it needs no masking
        const int min_valid = __reduce_min_sync(0xffffffffu, static_cast<unsigned>(valid));
        // P V of this group's previous step s_prev (tile j - 1) must be done
        // before O is rescaled.  Its ring slot's barrier is unambiguous then:
        // P V of step s_prev - 3 finished before S of step s (issued after
        // it), and P V of step s_prev + 3 > s cannot have been issued, as P V
        // goes in step order and that of step s needs this thread's P.
        const int s_prev = j > 0 ? g0 + sch.step(x, j - 1) : 0;
        float2 sum2 = make_float2(0.f, 0.f);
        // P of 32 keys = 16 columns (two 16-bit values each) over S columns
        // [16 c, 16 c + 16), which belong to S chunks already read
        auto store_p = [&](int c, const uint32_t(&pk)[16]) { tmem_st_32x32b_x16(lane_base + s_col + 16 * c, pk); };
        // x = s * scale - m for the 32 keys of a chunk (-inf for masked
        // keys), then p = exp2(x) on the SFU in fp32, rounded to the 16-bit
        // type into P, and their fp32 sum added to sum2.  A chunk whose
        // exponentials sum to more than 2^8 in some row is neither stored nor
        // summed, and the function returns false: every key above m + 8 (log2
        // units; a maximum that must be raised) is caught so, since its own
        // exponential is part of the sum, by one test on a sum the chunk
        // forms anyway (a test of each key against m + 8 took 16 more
        // instructions per chunk); a chunk caught without such a key is
        // recomputed with the same m below.  Four independent chains for the
        // sum keep the SFU fed.
        // kFull: every key of the tile visible to every row of the warp,
        // known at compile time (no masking code)
        auto softmax_chunk = [&](int c, const uint32_t(&cur)[32], bool check, auto full) -> bool {
          constexpr bool kFull = decltype(full)::value;
          const float2 sc = make_float2(scale_log2, scale_log2), nm = make_float2(-m_run, -m_run);
          float2 xv[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i)
            xv[i] = __ffma2_rn(make_float2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), sc, nm);
          if (!kFull && c * 32 + 32 > min_valid) {
  #pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (c * 32 + 2 * i >= valid) xv[i].x = -INFINITY;
              if (c * 32 + 2 * i + 1 >= valid) xv[i].y = -INFINITY;
            }
          }
          float2 sq[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          uint32_t pk[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 p = make_float2(ex2(xv[i].x), ex2(xv[i].y));
            sq[i & 3] = __fadd2_rn(sq[i & 3], p);
            pk[i] = pack2<T16>(p.x, p.y);
          }
          const float2 cs = __fadd2_rn(__fadd2_rn(sq[0], sq[1]), __fadd2_rn(sq[2], sq[3]));
          if (check && __any_sync(0xffffffffu, cs.x + cs.y > kRescaleSum)) return false;
          sum2 = __fadd2_rn(sum2, cs);
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
        // maximum of the first chunk's visible scores.  A chunk that may hold
        // a score above m + 8 (log2 units; a maximum that must be raised)
        // stops it, and the rest of the tile is done below with the maximum
        // raised where it must be.
        bool done = false;
        int fail = kTK / 32;  // the chunk that stopped the single pass
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
          // a full tile (all its keys visible to every row of the warp: n_live
          // is 4) runs a copy without the masking and live-chunk tests
          // (measured: 12 layers at B = 16, T = 1024 went 0.621 -> 0.610
          // ms); the chunks' indices stay compile-time constants (a loop
          // over chunk pairs, half the code, took 0.665 ms)
          auto chunk = [&](auto cc, auto full, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
            constexpr int c = decltype(cc)::value;
            constexpr bool kFull = decltype(full)::value;
            if (!go) return;
            if (!kFull && c >= n_live) {
              zero_chunk(c);
              return;
            }
            const bool next_live = kFull ? (c + 1 < kTK / 32) : (c + 1 < n_live);
            if (next_live) tmem_ld_32x32b_x32(lane_base + s_col + (c + 1) * 32, nxt);
            go = softmax_chunk(c, cur, true, full);
            if (!go) fail = c;
            if (next_live) tmem_ld_wait_regs(nxt);
          };
          static_assert(kTK == 128, "four chunks of 32 keys");
          using I0 = std::integral_constant<int, 0>;
          using I1 = std::integral_constant<int, 1>;
          using I2 = std::integral_constant<int, 2>;
          using I3 = std::integral_constant<int, 3>;
          if (all_full) {
            const std::true_type f;
            chunk(I0(), f, ra, rb);
            chunk(I1(), f, rb, ra);
            chunk(I2(), f, ra, rb);
            chunk(I3(), f, rb, ra);
          } else {
            const std::false_type f;
            chunk(I0(), f, ra, rb);
            chunk(I1(), f, rb, ra);
            chunk(I2(), f, ra, rb);
            chunk(I3(), f, rb, ra);
          }
          done = go;
        }
        if (!done) {
          // A maximum that grows by more than 2^8 in chunk `fail`: P of the
          // chunks before it is in TMEM (their scores are below m + 8, so the
          // new maximum comes from chunks fail..); their S columns are gone,
          // those of chunks fail.. are intact.  The row maximum over chunks
          // fail.., the rescale of O, of the sum and of the P already written,
          // then the exponentials of chunks fail...
          float mx = -INFINITY;
  #pragma unroll 1
          for (int c = fail; c < kTK / 32; ++c) {
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
            const float alpha = ex2(m_run - m_new);
            if (j > 0) {
              if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[s_prev % kRing], (s_prev / kRing) & 1))))
                break;
              tc_fence_after();
  #pragma unroll 1
              for (int c = 0; c < kHS / 32; ++c) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(lane_base + kTmemO + x * kHS + c * 32, o);
                tmem_ld_wait();
  #pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st_32x32b_x32(lane_base + kTmemO + x * kHS + c * 32, o);
              }
              l_run *= alpha;
            }
            tmem_st_wait();  // the P chunks written so far are readable
  #pragma unroll 1
            for (int c = 0; c < fail; ++c) {
              uint32_t pk[16];
              tmem_ld_32x32b_x16(lane_base + s_col + 16 * c, pk);
              tmem_ld_wait();
  #pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float2 v = unpack2<T16>(pk[e]);
                pk[e] = pack2<T16>(v.x * alpha, v.y * alpha);
              }
              store_p(c, pk);
            }
            sum2 = make_float2(sum2.x * alpha, sum2.y * alpha);
            m_run = m_new;
          }
  #pragma unroll 1
          for (int c = fail; c < kTK / 32; ++c) {
            uint32_t rr[32];
            tmem_ld_32x32b_x32(lane_base + s_col + c * 32, rr);
            tmem_ld_wait_regs(rr);
            softmax_chunk(c, rr, false, std::false_type());
          }
        }
        l_run += sum2.x + sum2.y;
        tmem_st_wait();  // P written by this thread is in TMEM before the MMA reads it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[r]);
        if (j == 0 && pend.k >= 0 && !(ok = epilogue(pend))) break;
      }
      if (!ok) break;
      if (pend.k >= 0 && !(ok = epilogue(pend))) break;  // no step of this group in this unit
      if (n_x > 0) {
        pend = Done{k, m_run, l_run};
        ++before;
      }
      g0 += sch.n_steps;
    }
    if (ok && pend.k >= 0) ok = epilogue(pend);
    if (!ok) *abort_flag = 1;
    if (lane == 0) bulk_wait_group_read<0>();  // the staging rows are read before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The units' table for G CTAs: units in their numbering (non-increasing
// length), each to the CTA with the least work so far, ties to the lowest
// CTA; a unit's work is its steps plus one (its first loads and its
// epilogue cost about a step).  No table (n = 0) past the table's size.
// Kept per thread for the last shape asked.
const UnitSchedule& unit_schedule(int B, int T, int NH, int G) {
  thread_local UnitSchedule sc{};
  thread_local int key[4] = {-1, -1, -1, -1};
  if (key[0] == B && key[1] == T && key[2] == NH && key[3] == G) return sc;
  key[0] = B;
  key[1] = T;
  key[2] = NH;
  key[3] = G;
  sc = UnitSchedule{};
  const int U = (T + 2 * kTQ - 1) / (2 * kTQ), per_u = B * NH, kv_tiles = (T + kTK - 1) / kTK;
  const long long n_units = static_cast<long long>(U) * per_u;
  if (G <= 0 || G > kSchedMaxCtas || n_units > kSchedMaxUnits) return sc;
  std::vector<std::vector<int>> lists(G);
  using Load = std::pair<long long, int>;  // (work so far, CTA)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> least;
  for (int c = 0; c < G; ++c) least.push({0, c});
  for (int k = 0; k < n_units; ++k) {
    const int u = U - 1 - k / per_u;
    const int n_a = std::min(2 * u + 1, kv_tiles);
    const int n_b = (2 * u + 1) * kTQ < T ? std::min(2 * u + 2, kv_tiles) : 0;
    const Load top = least.top();
    least.pop();
    lists[top.second].push_back(k);
    least.push({top.first + n_a + n_b + 1, top.second});
  }
  int e = 0;
  for (int c = 0; c < G; ++c) {
    sc.first[c] = static_cast<uint16_t>(e);
    for (int k : lists[c]) sc.unit[e++] = static_cast<uint16_t>(k);
  }
  sc.first[G] = static_cast<uint16_t>(e);
  sc.n = e;
  return sc;
}

template <typename T16, typename OutT>
int launch_typed(void* out, float* lse, const CUtensorMap& map, int B, int T, int C, int NH, cudaStream_t s) {
  // the output [B][T][C] as boxes of 128 bytes x 32 rows (one warp's rows),
  // 128-byte swizzle
  CUtensorMap map_out;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[2] = {static_cast<uint64_t>(C) * sizeof(OutT), static_cast<uint64_t>(T) * C * sizeof(OutT)};
    const uint32_t box[3] = {128 / static_cast<uint32_t>(sizeof(OutT)), 32, 1};  // 128-byte rows
    const CUtensorMapDataType dt = std::is_same<OutT, float>::value     ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : std::is_same<OutT, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_tensor_map(&map_out, dt, 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return GPT2_ERR_CUDA;
  }
  static bool attr_set[kMaxDevices] = {};  // per template instance and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  auto kern = attn_tc05_kernel<T16, OutT>;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  static int sms[kMaxDevices] = {};
  if (sms[dev] == 0) {
    const cudaError_t e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return note_cuda_error(e);
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  // persistent: one CTA per SM (at most one per unit)
  const long long units = static_cast<long long>((T + 2 * kTQ - 1) / (2 * kTQ)) * B * NH;
  if (units > 0x7fffffffLL) return GPT2_ERR_SHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < sms[dev] ? units : sms[dev]));
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Smem::alloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits for its predecessor itself
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_on() ? 1 : 0;
  const int Tp = (T + kTQ - 1) / kTQ * kTQ;
  const UnitSchedule& sched = unit_schedule(B, T, NH, static_cast<int>(cfg.gridDim.x));
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, map_out, lse, B, T, NH, Tp, scale_log2, sched);
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
