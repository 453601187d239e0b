// attention_bwd_tc.cu -- the backward pass of causal attention on the
// sm_103a tensor cores (tcgen05, TMEM, TMA), head size 64, bf16 operands
// and fp32 accumulation ("Understand FlashAttention (II)": the backward of
// Algorithm 1, P recomputed tile by tile from the forward's row statistic).
//
// With S = Q K^T / sqrt(64) (causal), P = softmax_rows(S), O = P V and the
// incoming gradient dO:
//   dV = P^T dO,  dP = dO V^T,  dS = P (dP - D),  D[t] = sum_d dO[t][d] O[t][d],
//   dQ = dS K / sqrt(64),  dK = dS^T Q / sqrt(64),
// and P = exp2(S log2(e) - L) from L = m + log2(l), the log-sum-exp of the
// forward's softmax in log2 units (written by the forward kernel).  The
// kernels compute P' = P / 8 = exp2(S log2(e) - L - 3) (L' = L + 3 is taken
// once, in the kernel that prepares D), so that dS' = P' (dP - D) is dS
// scaled by 1/sqrt(64) = 2^-3 with no multiply, and multiply dV by 8 once at
// the end (exact: powers of two).
//
// Two kernels, each a CTA (one per SM) over one 128-row tile of one
// (sequence, head), so that every gradient element is accumulated in one
// place and written once (no atomics; results do not depend on timing):
//   dK/dV  per key tile j: streams the query tiles i >= j (Q_i, dO_i and
//          their L and D), computes S^T = K Q_i^T and dP^T = V dO_i^T in
//          TMEM, P^T and dS^T (rows = keys) written back into TMEM over
//          the S^T and dP^T they came from, and accumulates dV += P^T dO_i
//          and dK += dS^T Q_i with those as A operands read from TMEM;
//   dQ     per query tile i: streams the key tiles j <= i (K_j, V_j),
//          computes S = Q K_j^T and dP = dO V_j^T, dS into TMEM over dP,
//          and accumulates dQ += dS K_j.
// In both, the "fixed" pair of tiles (K, V or Q, dO) stays in shared memory
// and the "streamed" pair (Q_i, dO_i or K_j, V_j) passes through a ring of
// three stages; the products are then uniform:
//   S  = fixed0 stream0^T,  dP = fixed1 stream1^T          (K-major operands)
//   dV += P^T stream1,  dK += dS^T stream0,  dQ += dS stream0   (stream tiles
//                                                    as MN-major B operands)
// Roles: warp 0 loads (TMA), warp 1 owns TMEM and issues the MMAs (one
// elected lane), warps 2-9 compute P and dS, one row per thread and half of
// the 128 columns per warp (two warps per TMEM lane quadrant).  TMEM: two S
// buffers (S of tile u + 2 is issued while tile u + 1 is processed), one dP
// buffer, the accumulators.  The softmax warps first turn S into P (kept
// in fp32 registers; stored as bf16 for dV), then wait for dP and form dS,
// so the dP product overlaps the exponentials.  The two warps of a TMEM
// lane quadrant share its lanes: each reads its half of the columns, and a
// 64-thread named barrier orders both reads before either writes P or dS
// over them (packed, the 128 columns of P fit in the first 64).  With P and
// dS in TMEM there are no shared-memory stores of them and no proxy fences
// (measured through shared memory: 64 KB of stores per tile pair).
// Every wait is bounded; a timeout sets the device error word and the CTA
// drains its copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

namespace gpt2 {
namespace {

constexpr int kR = 128;               // rows of a tile (keys or queries) = TMEM lanes
constexpr int kHS = 64;               // head size
constexpr int kTile = kR * kHS * 2;   // 16 KB: 128 rows of 128 bytes
constexpr int kStages = 3;
// Buffers of the fixed tiles: the S products run up to two tiles ahead,
// which with one-tile items reaches the item after next; with three buffers
// the one it needs was last used three items back, long released (with two
// it is the current item's, released only after the products that wait for
// it: a deadlock)
constexpr int kFixed = 3;
constexpr int kSmWarps = 8;
constexpr int kThreads = 64 + 32 * kSmWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;         // S buffers 0 and 1 (128 columns each)
constexpr uint32_t kTmemDP = 2 * kR;   // dP
constexpr uint32_t kTmemAcc = 3 * kR;  // dV (64 columns) then dK (64), or dQ (64)
constexpr uint32_t kIdescS = make_idesc(1u, kR, kR);                  // bf16, 128 x 128, both K-major
constexpr uint32_t kIdescAcc = make_idesc(1u, kR, kHS) | (1u << 16);  // 128 x 64, B MN-major

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kDQ>
struct BwdSmem {
  static constexpr int fixed = 0;                                 // kFixed buffers of two tiles
  static constexpr int stage = fixed + kFixed * 2 * kTile;        // kStages x two tiles
  static constexpr int stats = stage + kStages * 2 * kTile;       // dK/dV: kStages x (L'[128], D[128])
  static constexpr int bars = stats + (kDQ ? 0 : kStages * 2 * kR * 4);
  // fixed_full[kFixed], fixed_empty[kFixed]; st_full[kStages],
  // st_empty[kStages]; s_full[2]; dp_full, p_full, p_empty, ds_full,
  // acc_done, acc_free, drain
  static constexpr int n_bars = 2 * kFixed + 2 * kStages + 2 + 7;
  static constexpr int misc = bars + n_bars * 8;
  static constexpr int total = misc + 16;
  static constexpr int alloc = total + 1024;
};
static_assert(BwdSmem<false>::alloc <= 232448 && BwdSmem<true>::alloc <= 232448, "shared memory budget");

// D = A B^T over the 64 head dimensions: A, B K-major 128-row tiles
__device__ __forceinline__ void mma_dim(uint32_t d, uint32_t a_addr, uint32_t b_addr) {
  const uint64_t ad = smem_desc_sw128(a_addr), bd = smem_desc_sw128(b_addr);
#pragma unroll
  for (int kk = 0; kk < kHS / 16; ++kk)  // 16 dimensions = 32 bytes = 2 in the address field
    tc_mma_warp<false>(d, ad + 2 * kk, bd + 2 * kk, kIdescS, kk > 0 ? 1u : 0u);
}

// D (+)= A B over 128 rows: A a 128 x 128 bf16 operand in TMEM (rows in
// lanes, two values per column: 64 columns from a_tmem), B a 128-row tile
// read MN-major (64 contiguous head dimensions per row of K)
__device__ __forceinline__ void mma_rows(uint32_t d, uint32_t a_tmem, uint32_t b_addr, bool first) {
  const uint64_t bd = smem_desc_sw128_mn(b_addr, 1024);
#pragma unroll
  for (int kk = 0; kk < kR / 16; ++kk)  // A: 16 columns = 8 TMEM columns; B: 16 rows of 128 bytes
    tc_mma_ts_warp(d, a_tmem + kk * 8, bd + kk * (2048 / 16), kIdescAcc, (!first || kk > 0) ? 1u : 0u);
}

// Work items: a fixed tile of one (sequence, head), numbered by decreasing
// length (the number of streamed tiles), then b, then h; CTA c of G takes
// items c, 2G - 1 - c, 2G + c, ... (alternate rounds backwards).
template <bool kDQ>
struct BwdItems {
  int c, G, n_items, per, NH, n_tiles;
  __device__ int id(int i) const {
    const int k = i * G + ((i & 1) ? G - 1 - c : c);
    return k < n_items ? k : -1;
  }
  // dK/dV: key tile ft, streamed query tiles ft .. n_tiles - 1; dQ: query
  // tile ft, streamed key tiles 0 .. ft
  __device__ void get(int k, int& ft, int& b, int& h, int& n) const {
    const int r = k / per, bh = k % per;
    b = bh / NH;
    h = bh % NH;
    ft = kDQ ? n_tiles - 1 - r : r;
    n = kDQ ? ft + 1 : n_tiles - ft;
  }
  __device__ int length(int k) const { return n_tiles - k / per; }  // longest first: r = 0 streams all tiles
};

// A position in a CTA's sequence of streamed tiles over its items: item i
// (list index), its tile u of n, and the tiles before the item (g0).
template <bool kDQ>
struct BwdCursor {
  const BwdItems<kDQ>* it;
  int i, k, u, g0, n;
  __device__ explicit BwdCursor(const BwdItems<kDQ>* items) : it(items), i(0), u(0), g0(0), n(0) {
    k = it->id(0);
    if (k >= 0) n = it->length(k);
  }
  __device__ bool valid() const { return k >= 0; }
  __device__ int g() const { return g0 + u; }
  __device__ void advance() {
    if (++u < n) return;
    g0 += n;
    u = 0;
    k = it->id(++i);
    if (k >= 0) n = it->length(k);
  }
};

// kDQ = false: the dK/dV kernel; kDQ = true: the dQ kernel.  Persistent:
// one CTA per SM over its items, the fixed tiles of the next item loading
// into a second buffer, the streamed tiles' ring and the TMEM buffers
// continuing across items (measured: a CTA per item spent about 5800 cycles
// before its first S).  qkv map: [B][T][3C] bf16, do map: [B][T][C] bf16,
// boxes of 64 x 128 with the 128-byte swizzle.  Lse (L + 3), Dv:
// [B][NH][Tp] fp32, Tp = T rounded up to 128, zero past T.
template <bool kDQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc05_kernel(const __grid_constant__ CUtensorMap tmap_qkv, const __grid_constant__ CUtensorMap tmap_do,
                         float* __restrict__ dqkv, const float* __restrict__ Lse, const float* __restrict__ Dv, int B,
                         int T, int NH, int Tp, float scale_log2) {
  using L = BwdSmem<kDQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* fixed_full = bars;                  // [kFixed] the fixed tiles of item i (buffer i % kFixed) landed
  uint64_t* fixed_empty = fixed_full + kFixed;  // [kFixed] item i's products have read them
  uint64_t* st_full = fixed_empty + kFixed;     // [kStages] a streamed tile pair (and its L, D) landed
  uint64_t* st_empty = st_full + kStages;  // [kStages] its last reader is done
  uint64_t* s_full = st_empty + kStages;   // [2] S of tile g in buffer g % 2
  uint64_t* dp_full = s_full + 2;          // dP of tile g (phase g % 2)
  uint64_t* p_full = dp_full + 1;          // the P warps have written P^T of tile g into TMEM (dK/dV)
  // dV of tile g is done (dK/dV): the P warps wait for it before writing P^T
  // of tile g + 1, so that p_full is never two phases ahead of the MMA warp
  // (P^T of g + 1 needs only S of g + 1, issued before dV of g)
  uint64_t* p_empty = p_full + 1;
  uint64_t* ds_full = p_empty + 1;         // ... read dP and written dS of tile g into TMEM
  uint64_t* acc_done = ds_full + 1;        // item i's accumulators are final (phase i % 2)
  uint64_t* acc_free = acc_done + 1;       // ... and read by the epilogue
  uint64_t* drain = acc_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = NH * kHS;
  BwdItems<kDQ> items;
  items.c = blockIdx.x;
  items.G = gridDim.x;
  items.NH = NH;
  items.per = B * NH;
  items.n_tiles = (T + kR - 1) / kR;
  items.n_items = items.n_tiles * items.per;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kFixed; ++i) {
      mbar_init(&fixed_full[i], 1u);
      mbar_init(&fixed_empty[i], 1u);
    }
    mbar_init(&s_full[0], 1u);
    mbar_init(&s_full[1], 1u);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&st_full[i], 1u);
      mbar_init(&st_empty[i], 1u);
    }
    mbar_init(dp_full, 1u);
    mbar_init(p_full, kSmWarps);
    mbar_init(p_empty, 1u);
    mbar_init(ds_full, kSmWarps);
    mbar_init(acc_done, 1u);
    mbar_init(acc_free, kSmWarps);
    mbar_init(drain, 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_qkv);
    tma_prefetch_desc(&tmap_do);
  }
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
      uint32_t filled = 0, par = 0;    // per stage: ever filled; parity of the last fill
      uint32_t ffilled = 0, fpar = 0;  // the same per fixed buffer
      int f = 0;                       // streamed tile pairs loaded so far
      for (int i = 0;; ++i) {
        const int k = items.id(i);
        if (k < 0 || *abort_flag) break;
        int ft, b, h, n;
        items.get(k, ft, b, h, n);
        const size_t bh = static_cast<size_t>(b) * NH + h;
        // fixed: K_j, V_j (dK/dV) or Q_i, dO_i (dQ), into buffer i % kFixed
        // once item i - kFixed's products have read it
        const int fb = i % kFixed;
        const uint32_t fph = (i / kFixed) & 1;
        if (!mbar_wait(&fixed_empty[fb], fph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* fdst = smem + L::fixed + fb * 2 * kTile;
        mbar_arrive_expect_tx(&fixed_full[fb], 2 * kTile);
        if (!kDQ) {
          tma_load_3d(fdst, &tmap_qkv, &fixed_full[fb], C + h * kHS, ft * kR, b);
          tma_load_3d(fdst + kTile, &tmap_qkv, &fixed_full[fb], 2 * C + h * kHS, ft * kR, b);
        } else {
          tma_load_3d(fdst, &tmap_qkv, &fixed_full[fb], h * kHS, ft * kR, b);
          tma_load_3d(fdst + kTile, &tmap_do, &fixed_full[fb], h * kHS, ft * kR, b);
        }
        ffilled |= 1u << fb;
        fpar = (fpar & ~(1u << fb)) | (fph << fb);
        bool ok = true;
        for (int u = 0; u < n; ++u, ++f) {
          const int st = f % kStages;
          const uint32_t ph = (f / kStages) & 1;
          if (!mbar_wait(&st_empty[st], ph ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + L::stage + st * 2 * kTile;
          if (!kDQ) {  // Q_i, dO_i, L' and D of query tile i
            const int qi = ft + u;
            mbar_arrive_expect_tx(&st_full[st], 2 * kTile + 2 * kR * 4);
            tma_load_3d(dst, &tmap_qkv, &st_full[st], h * kHS, qi * kR, b);
            tma_load_3d(dst + kTile, &tmap_do, &st_full[st], h * kHS, qi * kR, b);
            float* sd = reinterpret_cast<float*>(smem + L::stats) + st * 2 * kR;
            bulk_load(sd, Lse + bh * Tp + static_cast<size_t>(qi) * kR, kR * 4, &st_full[st]);
            bulk_load(sd + kR, Dv + bh * Tp + static_cast<size_t>(qi) * kR, kR * 4, &st_full[st]);
          } else {  // K_j, V_j
            mbar_arrive_expect_tx(&st_full[st], 2 * kTile);
            tma_load_3d(dst, &tmap_qkv, &st_full[st], C + h * kHS, u * kR, b);
            tma_load_3d(dst + kTile, &tmap_qkv, &st_full[st], 2 * C + h * kHS, u * kR, b);
          }
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
      for (int fb = 0; fb < kFixed; ++fb)
        if ((ffilled >> fb) & 1u) mbar_wait(&fixed_full[fb], (fpar >> fb) & 1u);
      for (int st = 0; st < kStages; ++st)
        if ((filled >> st) & 1u) mbar_wait(&st_full[st], (par >> st) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    // The CTA's tiles in one sequence over its items: a cursor for S (two
    // tiles ahead), one for dP (one ahead), one for the gradient products.
    auto fixed0 = [&](int i) { return smem_u32(smem + L::fixed + (i % kFixed) * 2 * kTile); };
    auto stream0 = [&](int f) { return smem_u32(smem + L::stage + (f % kStages) * 2 * kTile); };
    // S of the cursor's tile into buffer g % 2 (the item's first waits for
    // its fixed tiles; every S waits for its streamed pair)
    auto issue_s = [&](const BwdCursor<kDQ>& c) -> bool {
      const int g = c.g();
      if (c.u == 0 && !__all_sync(0xffffffffu, mbar_wait(&fixed_full[c.i % kFixed], (c.i / kFixed) & 1)))
        return false;
      if (!__all_sync(0xffffffffu, mbar_wait(&st_full[g % kStages], (g / kStages) & 1))) return false;
      tc_fence_after();
      mma_dim(tmem + kTmemS + (g & 1) * kR, fixed0(c.i), stream0(g));
      tc_commit_warp(&s_full[g & 1]);
      return true;
    };
    // dP of the cursor's tile (its S, issued earlier, waited for its loads)
    auto issue_dp = [&](const BwdCursor<kDQ>& c) {
      const int g = c.g();
      mma_dim(tmem + kTmemDP, fixed0(c.i) + kTile, stream0(g) + kTile);
      tc_commit_warp(dp_full);
    };
    BwdCursor<kDQ> cs(&items), cd(&items);
    bool ok = true;
    if (cs.valid()) {
      ok = issue_s(cs);
      cs.advance();
    }
    if (ok && cd.valid()) {
      issue_dp(cd);
      cd.advance();
    }
    if (ok && cs.valid()) {
      ok = issue_s(cs);
      cs.advance();
    }
    for (BwdCursor<kDQ> c(&items); c.valid() && ok; c.advance()) {
      const int g = c.g();
      // the item's first gradient product overwrites the accumulators: the
      // previous item's epilogue must have read them
      if (c.u == 0 && c.i > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(acc_free, (c.i - 1) & 1)))) break;
      if (!kDQ) {
        // dV += P'^T dO_i once P^T is in TMEM over S^T of tile g; S two tiles
        // on then goes into that buffer (the products run in issue order)
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(p_full, g & 1)))) break;
        tc_fence_after();
        mma_rows(tmem + kTmemAcc, tmem + kTmemS + (g & 1) * kR, stream0(g) + kTile, c.u == 0);
        tc_commit_warp(p_empty);
        if (cs.valid()) {
          if (!(ok = issue_s(cs))) break;
          cs.advance();
        }
      }
      // dS in TMEM over dP: dK += dS^T Q_i (or dQ += dS K_j), then dP of the
      // next tile into the same columns (issued after: the products run in
      // issue order)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(ds_full, g & 1)))) break;
      tc_fence_after();
      mma_rows(tmem + kTmemAcc + (kDQ ? 0 : kHS), tmem + kTmemDP, stream0(g), c.u == 0);
      tc_commit_warp(&st_empty[g % kStages]);
      if (c.u == c.n - 1) {
        tc_commit_warp(acc_done);
        tc_commit_warp(&fixed_empty[c.i % kFixed]);
      }
      if (cd.valid()) {
        issue_dp(cd);
        cd.advance();
      }
      if (kDQ && cs.valid()) {  // S of tile g was read before dS was formed
        if (!(ok = issue_s(cs))) break;
        cs.advance();
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
    tc_commit_warp(drain);
    mbar_wait(drain, 0);
  } else {
    // ------------------------------------------------------- P and dS
    const int sw = warp - 2;
    const int qw = warp & 3;        // TMEM lane quadrant this warp may access
    const int hf = sw >> 2;         // columns [64 hf, 64 hf + 64)
    const int row = qw * 32 + lane; // row of the tile = TMEM lane
    const int col0 = hf * 64;
    const int pair_bar = 1 + qw;    // the named barrier of this quadrant's two warps
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    bool ok = true;
    int g0 = 0;  // tiles of the items before this one
    for (int i = 0; ok; ++i) {
      const int k = items.id(i);
      if (k < 0) break;
      int ft, b, h, n;
      items.get(k, ft, b, h, n);
      const size_t bh = static_cast<size_t>(b) * NH + h;
      const int f0 = g0;  // the streamed pairs run with the tiles
      float l_row = 0.f, d_row = 0.f;  // dQ kernel: the row's L' and D
      if (kDQ) {
        const size_t at = bh * Tp + static_cast<size_t>(ft) * kR + row;
        l_row = __ldg(Lse + at);
        d_row = __ldg(Dv + at);
      }
      for (int u = 0; u < n && ok; ++u) {
        const int g = g0 + u, f = f0 + u;  // this tile's place in the CTA's sequence
        const int sb = g & 1;
        bool got = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (g >> 1) & 1));
        const float* stats = nullptr;  // dK/dV: L' and D of the query tile, per column
        if (!kDQ) {
          // (complete already: S of tile u was issued after it)
          got = __all_sync(0xffffffffu, got && mbar_wait(&st_full[f % kStages], (f / kStages) & 1));
          stats = reinterpret_cast<const float*>(smem + L::stats) + (f % kStages) * 2 * kR;
        }
        // visible columns [lo, hi) of this row
        int lo, hi;
        if (!kDQ) {  // row = key ft * 128 + row; column = query (ft + u) * 128 + c: c >= row on the diagonal, < T
          lo = u == 0 ? row : 0;
          hi = min(T - (ft + u) * kR, kR);
        } else {  // row = query ft * 128 + row; column = key u * 128 + c <= query
          lo = 0;
          hi = max(0, min(ft * kR + row - u * kR + 1, kR));
        }
        const bool all_valid = lo <= col0 && hi >= col0 + 64;
        uint32_t sv[2][32];
        if (got) {
          tc_fence_after();
          tmem_ld_32x32b_x32(lane_base + kTmemS + sb * kR + col0, sv[0]);
          tmem_ld_32x32b_x32(lane_base + kTmemS + sb * kR + col0 + 32, sv[1]);
          tmem_ld_wait();
        }
        // both warps of the quadrant have read their S columns (or one gave up)
        if (bar_or(pair_bar, 64, !got)) {
          ok = false;
          break;
        }
        // P' = exp2(S log2(e)/8 - L'), zero outside [lo, hi); kept in sv as fp32
        const float2 sc = make_float2(scale_log2, scale_log2);
  #pragma unroll
        for (int c = 0; c < 2; ++c) {
  #pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 nl4;
            if (kDQ) {
              nl4 = make_float4(-l_row, -l_row, -l_row, -l_row);
            } else {
              const float4 lv = *reinterpret_cast<const float4*>(stats + col0 + c * 32 + e);
              nl4 = make_float4(-lv.x, -lv.y, -lv.z, -lv.w);
            }
            float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), sc,
                                   make_float2(nl4.x, nl4.y));
            float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3])), sc,
                                   make_float2(nl4.z, nl4.w));
            if (!all_valid) {
              const int cc = col0 + c * 32 + e;
              if (cc < lo || cc >= hi) x0.x = -INFINITY;
              if (cc + 1 < lo || cc + 1 >= hi) x0.y = -INFINITY;
              if (cc + 2 < lo || cc + 2 >= hi) x1.x = -INFINITY;
              if (cc + 3 < lo || cc + 3 >= hi) x1.y = -INFINITY;
            }
            sv[c][e] = __float_as_uint(ex2(x0.x));
            sv[c][e + 1] = __float_as_uint(ex2(x0.y));
            sv[c][e + 2] = __float_as_uint(ex2(x1.x));
            sv[c][e + 3] = __float_as_uint(ex2(x1.y));
          }
        }
        bool p_ok = true;
        if (!kDQ) {
          // P'^T (bf16 pairs) over this warp's half of the first 64 columns of
          // S^T's buffer: the A operand of dV (once dV of the CTA's previous
          // tile is done: p_empty)
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(sv[e >> 4][(e & 15) * 2]), __uint_as_float(sv[e >> 4][(e & 15) * 2 + 1]));
          if (g > 0) p_ok = __all_sync(0xffffffffu, mbar_wait(p_empty, (g - 1) & 1));
          if (p_ok) {
            tmem_st_32x32b_x32(lane_base + kTmemS + sb * kR + hf * 32, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
          }
        }
        // dS' = P' (dP - D), one 32-column chunk of dP at a time; the second
        // chunk's load completes this warp's reads of dP before the barrier
        // (a wait given up above reaches the quadrant's barrier below as a failure)
        got = p_ok && __all_sync(0xffffffffu, mbar_wait(dp_full, g & 1));
        if (got) tc_fence_after();
        uint32_t pk[32];
        bool gave_up = false;
  #pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dv[32];
          if (got) {
            tmem_ld_32x32b_x32(lane_base + kTmemDP + col0 + c * 32, dv);
            tmem_ld_wait();
          }
          if (c == 1 && bar_or(pair_bar, 64, !got)) {  // both warps of the quadrant have read their dP
            gave_up = true;
            break;
          }
  #pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 d4;
            if (kDQ) {
              d4 = make_float4(d_row, d_row, d_row, d_row);
            } else {
              d4 = *reinterpret_cast<const float4*>(stats + kR + col0 + c * 32 + e);
            }
            const float2 g0 = __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                         make_float2(-d4.x, -d4.y));
            const float2 g1 = __fadd2_rn(make_float2(__uint_as_float(dv[e + 2]), __uint_as_float(dv[e + 3])),
                                         make_float2(-d4.z, -d4.w));
            const float2 q0 = __fmul2_rn(make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), g0);
            const float2 q1 = __fmul2_rn(make_float2(__uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3])), g1);
            pk[c * 16 + e / 2] = pack_bf16x2(q0.x, q0.y);
            pk[c * 16 + e / 2 + 1] = pack_bf16x2(q1.x, q1.y);
          }
        }
        if (gave_up) {
          ok = false;
          break;
        }
        tmem_st_32x32b_x32(lane_base + kTmemDP + hf * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
      if (!ok) break;
      // both warps of the quadrant agree on the outcome before either goes
      // on to the next item's barriers
      const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(acc_done, i & 1));
      if (bar_or(pair_bar, 64, !acc_ok)) {
        ok = false;
        break;
      }
      {
        tc_fence_after();
        // dK/dV: warps of half 0 write dV, half 1 dK (64 columns each); dQ:
        // each half 32 of dQ's columns
        const int r_glob = ft * kR + row;
        const int n_chunks = kDQ ? 1 : 2;
        const uint32_t t_col = kTmemAcc + (kDQ ? hf * 32 : hf * kHS);
        const int g_col = kDQ ? h * kHS + hf * 32 : (hf == 0 ? 2 * C : C) + h * kHS;
  #pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(lane_base + t_col + c * 32, o);
          tmem_ld_wait();
          if (r_glob < T) {
            float* dst = dqkv + (static_cast<size_t>(b) * T + r_glob) * 3 * C + g_col + c * 32;
            const float f = (!kDQ && hf == 0) ? 8.0f : 1.0f;  // dV accumulated P' = P / 8
  #pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4*>(dst)[q] =
                  make_float4(__uint_as_float(o[4 * q]) * f, __uint_as_float(o[4 * q + 1]) * f,
                              __uint_as_float(o[4 * q + 2]) * f, __uint_as_float(o[4 * q + 3]) * f);
          }
        }
        // the accumulators have been read: the next item may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
      }
      g0 += n;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dO [B,T,C] fp32 -> bf16 copy; D[b][h][t] = sum over the head's 64
// columns of dO * O; the forward's L becomes L' = L + 3 in place (the
// backward kernels compute P / 8); D and L' are zero for t in [T, Tp).
// Eight threads per head and row, eight columns each.
__global__ void attn_bwd_prep_kernel(__nv_bfloat16* __restrict__ do16, float* __restrict__ Dv, float* __restrict__ Lse,
                                     const float* __restrict__ dout, const float* __restrict__ out, int B, int T, int C,
                                     int NH, int Tp) {
  const long long per_row = C / 8;
  const long long total = static_cast<long long>(B) * Tp * per_row;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool live = idx < total;
  const long long r = live ? idx / per_row : 0;
  const int c8 = live ? static_cast<int>(idx % per_row) : 0;
  const int b = static_cast<int>(r / Tp), t = static_cast<int>(r % Tp);
  float dot = 0.f;
  if (live && t < T) {
    const size_t at = (static_cast<size_t>(b) * T + t) * C + c8 * 8;
    const float4 g0 = *reinterpret_cast<const float4*>(dout + at), g1 = *reinterpret_cast<const float4*>(dout + at + 4);
    const float4 o0 = *reinterpret_cast<const float4*>(out + at), o1 = *reinterpret_cast<const float4*>(out + at + 4);
    dot = g0.x * o0.x + g0.y * o0.y + g0.z * o0.z + g0.w * o0.w + g1.x * o1.x + g1.y * o1.y + g1.z * o1.z +
          g1.w * o1.w;
    *reinterpret_cast<uint4*>(do16 + at) =
        make_uint4(pack_bf16x2(g0.x, g0.y), pack_bf16x2(g0.z, g0.w), pack_bf16x2(g1.x, g1.y), pack_bf16x2(g1.z, g1.w));
  }
  // the eight threads of a head are eight aligned lanes of one warp
  dot += __shfl_xor_sync(0xffffffffu, dot, 1);
  dot += __shfl_xor_sync(0xffffffffu, dot, 2);
  dot += __shfl_xor_sync(0xffffffffu, dot, 4);
  if (live && (c8 & 7) == 0) {
    const size_t at = (static_cast<size_t>(b) * NH + c8 / 8) * Tp + t;
    Dv[at] = dot;
    Lse[at] = t < T ? Lse[at] + 3.0f : 0.f;
  }
}

template <bool kDQ>
int set_smem_attr() {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc05_kernel<kDQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               BwdSmem<kDQ>::alloc);
    if (e != cudaSuccess) return note_cuda_error(e);
    attr_set[dev] = true;
  }
  return GPT2_OK;
}

}  // namespace

int attn_bwd_padded_len(int T) { return (T + kR - 1) / kR * kR; }

void launch_attn_bwd_prep(void* do16, float* Dv, float* Lse, const float* dout, const float* out, int B, int T, int C,
                          int NH, cudaStream_t s) {
  const int Tp = attn_bwd_padded_len(T);
  const long long total = static_cast<long long>(B) * Tp * (C / 8);
  const int threads = 256;
  attn_bwd_prep_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, s>>>(
      static_cast<__nv_bfloat16*>(do16), Dv, Lse, dout, out, B, T, C, NH, Tp);
}

int launch_attention_backward_tc05(float* dqkv, const void* qkv16, const void* do16, const float* Lse,
                                   const float* Dv, int B, int T, int C, int NH, cudaStream_t s) {
  if (C / NH != kHS || C % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  int rc = set_smem_attr<false>();
  if (rc == GPT2_OK) rc = set_smem_attr<true>();
  if (rc != GPT2_OK) return rc;
  CUtensorMap map_qkv, map_do;
  const uint32_t box[3] = {kHS, kR, 1};
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(3 * C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[2] = {static_cast<uint64_t>(3 * C) * 2, static_cast<uint64_t>(T) * 3 * C * 2};
    if (!encode_tensor_map(&map_qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, qkv16, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return GPT2_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(C), static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[2] = {static_cast<uint64_t>(C) * 2, static_cast<uint64_t>(T) * C * 2};
    if (!encode_tensor_map(&map_do, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, do16, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return GPT2_ERR_CUDA;
  }
  const int Tp = attn_bwd_padded_len(T);
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  // persistent: one CTA per SM (at most one per item)
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
  if (sms[dev] == 0) {
    const cudaError_t e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return note_cuda_error(e);
  }
  const long long n_items = static_cast<long long>((T + kR - 1) / kR) * B * NH;
  if (n_items > 0x7fffffffLL) return GPT2_ERR_SHAPE;
  const dim3 grid(static_cast<unsigned>(n_items < sms[dev] ? n_items : sms[dev]));
  attn_bwd_tc05_kernel<false><<<grid, kThreads, BwdSmem<false>::alloc, s>>>(map_qkv, map_do, dqkv, Lse, Dv, B, T, NH,
                                                                            Tp, scale_log2);
  attn_bwd_tc05_kernel<true><<<grid, kThreads, BwdSmem<true>::alloc, s>>>(map_qkv, map_do, dqkv, Lse, Dv, B, T, NH,
                                                                          Tp, scale_log2);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GPT2_OK : note_cuda_error(e);
}

}  // namespace gpt2
