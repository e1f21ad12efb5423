// Forward kernel: O = softmax(Q K^T * scale) V for every (b, h) head, plus lse.
//
// "Attention Is All You Need", §3.2.1 eq. (1) and Figure 2 (MatMul, Scale,
// Mask (opt.), SoftMax, MatMul), with the decoder mask of §3.2.3. The paper
// runs eq. (1) as plain matrix multiplies on P100s; here both products run on
// the tcgen05 tensor cores and the softmax is streamed over key tiles with a
// running maximum, so the n x m weight matrix never leaves the SM.
//
// One CTA owns NQ query tiles of 128 rows of one head and streams BN-key
// tiles K_j, V_j through a TMA/mbarrier ring:
//   warp 4*NQ          TMA producer: the Q tiles once, then K_j and V_j per stage.
//   warp 4*NQ + 1 + g  MMA issuer of query tile g (one lane): S_g = Q_g K_j^T
//                      into TMEM, then O_g += P_g V_j with P_g read from TMEM.
//   warps 4g..4g+3     softmax of query tile g, one thread per row: load the S
//                      row from TMEM, row max, p = 2^(s*c - m) with
//                      c = scale*log2(e), row sum, bf16 P back into TMEM,
//                      rescale of the O row when the running max grew by more
//                      than 2^8, and finally O / l and lse.
// Each query tile has its own issuing thread. A thread that waits on an
// mbarrier stops feeding the tensor pipe, whose queue holds only a few MMAs;
// with one issuer per tile the other tiles' products fill those gaps, and the
// tiles run out of step, so one softmax group works while the tensor cores
// run the other group's products.
//
// Where TMEM has room (d <= 64 with 128-key tiles) P_g gets columns of its
// own: the softmax releases S_g as soon as the row is in registers, and
// S_g(j+1) is computed while the softmax of tile j still runs; the softmax
// waits for PV_g(j-1) only before it overwrites P_g. Otherwise P_g aliases
// S_g and the issue order per tile is PV_g(j), S_g(j+1); the commit that
// signals S_g(j+1) then also proves that PV_g(j) finished. Either way the O
// rescale of tile j runs after PV_g(j-1) and before PV_g(j). With the causal
// mask only the key tiles at or below the diagonal are loaded and multiplied.
//
// TMEM columns: S_g at [g*BN, (g+1)*BN); with separate P, P_g (bf16 pairs) at
// NQ*BN + g*BN/2; O_g after them, D columns each.
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr float kLn2 = 0.69314718055994530942f;
// Speculative exponentials (persistent forward): a tile is exponentiated against
// the running reference without taking its own maximum first; a tile row whose
// weights sum above 2^8 is redone against its maximum. So no weight exceeds
// 2^8, the same bound the lazy rescale (threshold kRescaleThreshold = 8) keeps.
constexpr float kSpecLimitSum = 256.f;
// A stale running max is kept while new scores exceed it by at most 8 in
// log2 units (p <= 256), so most tiles skip the O rescale. Exact after the
// final division by the row sum.
constexpr float kRescaleThreshold = 8.0f;

constexpr uint32_t tmem_cols_for(uint32_t c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

// The O correction after a row's reference maximum moved: O = alpha * O in
// TMEM. It is rare once a row has seen a few key tiles, and it stays out of
// line so that the softmax loops do not carry its registers and code (inlined,
// the never-taken branch cost 5 % at n = m = 16384, d = 64).
template <int NCOL>
__device__ __noinline__ void rescale_o(uint32_t t_o, float alpha) {
#pragma unroll
  for (int q = 0; q < NCOL / 16; ++q) {
    uint32_t o[16];
    tmem_ld16(t_o + q * 16, o);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
    tmem_st16(t_o + q * 16, o);
  }
}

template <int D, int NQ, int BN>
struct Fwd {
  // P in TMEM columns of its own (see above)
  static constexpr bool SEP_P = (D <= 64 && BN == 128 && NQ * (BN + BN / 2 + D) <= 512);
  static constexpr uint32_t P_COLS = SEP_P ? BN / 2 : 0;
  static_assert(NQ * (BN + P_COLS + D) <= 512, "TMEM holds at most 512 fp32 columns");
  static constexpr int ATOM = (D >= 64) ? 64 : D;        // bf16 elements per swizzle row
  static constexpr int NATOM = D / ATOM;                  // TMA boxes per tile
  static constexpr uint32_t SWZ = (D >= 64) ? 2u : 4u;    // descriptor code: 128B / 64B swizzle
  static constexpr uint32_t SBO = 8u * ATOM * 2u;         // bytes between 8-row groups
  static constexpr uint32_t QTILE = 128u * D * 2u;        // one 128-row query tile
  static constexpr uint32_t QBOX = 128u * ATOM * 2u;
  static constexpr uint32_t KTILE = BN * D * 2u;          // one key (or value) tile
  static constexpr uint32_t KBOX = BN * ATOM * 2u;
  static constexpr int STAGES = (NQ * QTILE + 4 * 2 * KTILE <= 200u * 1024u) ? 4
                                : (NQ * QTILE + 3 * 2 * KTILE <= 200u * 1024u) ? 3 : 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = NQ * QTILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KTILE;
  static constexpr uint32_t TMEM_COLS = tmem_cols_for(NQ * (BN + P_COLS + D));
  static constexpr int MIN_BLOCKS = (TMEM_COLS <= 256 && OFF_V + STAGES * KTILE + 1024 <= 110u * 1024u) ? 2 : 1;
  // One softmax thread per query row (a variant with two threads per row,
  // half of the key columns each, measured slower on GB300: exchanging the
  // row maxima cost more than the shorter rows saved).
  static constexpr int COLS = BN;                         // key columns per softmax thread
  static constexpr int OCOLS = D;                         // O columns per softmax thread
  static constexpr uint32_t SMEM = OFF_V + STAGES * KTILE + 1024;  // + alignment slack
  static constexpr int SOFT_WARPS = 4 * NQ;
  // Softmax warpgroups, then one warpgroup with the producer, the NQ issuer
  // warps and idle padding, so that setmaxnreg can move registers from it to
  // the softmax warpgroups.
  static_assert(NQ + 1 <= 4, "producer and issuers share one warpgroup");
  static constexpr int THREADS = SOFT_WARPS * 32 + 128;
  static constexpr int REG_LAUNCH = (65536 / (THREADS * MIN_BLOCKS)) / 8 * 8;
  static constexpr int REG_OTHER = (MIN_BLOCKS == 2) ? 40 : 96;
  static constexpr int REG_SOFTMAX = ((THREADS * REG_LAUNCH - 128 * REG_OTHER) / (SOFT_WARPS * 32)) / 8 * 8;
  static_assert(REG_SOFTMAX * SOFT_WARPS * 32 + REG_OTHER * 128 <= THREADS * REG_LAUNCH,
                "register split exceeds the launch allocation");
  // a single CTA per SM with one thread per row has registers enough without a split
  static constexpr bool REG_SPLIT = (MIN_BLOCKS == 2);
  static constexpr int PRODUCER = SOFT_WARPS, ISSUER = SOFT_WARPS + 1;  // issuers: ISSUER .. ISSUER + NQ - 1
  static constexpr int CHUNKS = COLS / 32;                // 32-column TMEM loads per row
  __host__ __device__ static constexpr uint32_t tm_s(int g) { return g * BN; }
  __host__ __device__ static constexpr uint32_t tm_p(int g) { return SEP_P ? NQ * BN + g * P_COLS : g * BN; }
  __host__ __device__ static constexpr uint32_t tm_o(int g) { return NQ * (BN + P_COLS) + g * D; }
};

constexpr int kMaxNQ = 4;
constexpr int kMaxStages = 5;

struct FwdShared {
  uint64_t q_full;
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxNQ][kMaxStages];  // released by each query tile's issuer
  uint64_t s_full[kMaxNQ], p_full[kMaxNQ], o_full[kMaxNQ];
  uint64_t s_free[kMaxNQ], pv_done[kMaxNQ];  // separate P only
  uint64_t exp_turn[2];  // two query tiles: their exponential phases alternate
  uint64_t o_staged[kMaxNQ];
  uint64_t drain[kMaxNQ];
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A query row of a sequence without real keys (key padding with length 0):
// O = 0 and lse = -inf, the empty sum. Written directly; this case is rare.
template <int D>
__device__ __forceinline__ void write_empty_row(const FwdParams& p, int bh, int row, int col0, int ncols,
                                                bool write_lse) {
  if (row >= p.n) return;
  uint4* orow = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.n + row) * D + col0);
  for (int c = 0; c < ncols / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
  if (write_lse && p.lse != nullptr) p.lse[static_cast<size_t>(bh) * p.n + row] = -INFINITY;
}

// Key tiles of BN needed by query rows up to r_hi (already clipped to n-1).
template <int BN>
__device__ __forceinline__ int key_tiles(int r_hi, int m, int causal) {
  const int kv_hi = causal ? min(r_hi, m - 1) : (m - 1);
  return kv_hi / BN + 1;
}

// Waits without looking at the abort flag: used to let copies and MMAs that
// are already in flight finish before the CTA releases its resources.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

// p = 2^(s*c - m) for one 32-column chunk of a row held in registers; packs
// the bf16 weights into pk and adds the weights into lsum. MASKED: columns at
// or past `rem` or before `rlo` (keys this row may not see) get weight exactly 0
// (needed for c = 0 only: otherwise their scores hold -inf already).
// EXACT_SUM: the weights are added as rounded to bf16 (mixed-precision adds),
// so the row sum l is the sum of the weights the P.V product applies and O / l
// is an exact convex combination of value rows (a row dominated by one key
// returns that value row even when the reference m lags the row maximum).
// Otherwise the fp32 weights are added in pairs (one packed add per two
// weights): on GB300 the exp unit bounds this loop, and the mixed-precision
// adds take 30 % of its throughput (1.79 k against 1.38 k clocks per 128-key
// tile for two warps per scheduler, measured in isolation). The two sums
// differ by the bf16 rounding of the weights, relative 2^-9 at most; only
// rows that one key dominates see it in O.
template <bool MASKED, bool EXACT_SUM>
__device__ __forceinline__ void exp_chunk(const uint32_t (&s)[32], int col0, int rlo, int rem, uint64_t c2,
                                          uint64_t nm2, float (&lsum)[4], uint32_t (&pk)[16]) {
  uint64_t acc[2];
  if (!EXACT_SUM) {
    acc[0] = f2_pack(lsum[0], lsum[1]);
    acc[1] = f2_pack(lsum[2], lsum[3]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t x2 = fma2(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, nm2);
    float x0, x1;
    f2_unpack(x2, x0, x1);
    if (MASKED) {
      if (col0 + 2 * i >= rem || col0 + 2 * i < rlo) x0 = -INFINITY;
      if (col0 + 2 * i + 1 >= rem || col0 + 2 * i + 1 < rlo) x1 = -INFINITY;
    }
    const uint64_t p2 = f2_pack(ex2(x0), ex2(x1));
    pk[i] = pack_bf16x2_pair(p2);
    if (EXACT_SUM) acc_bf16x2(lsum[(i & 1) * 2], lsum[(i & 1) * 2 + 1], pk[i]);
    else acc[i & 1] = add2(acc[i & 1], p2);
  }
  if (!EXACT_SUM) {
    f2_unpack(acc[0], lsum[0], lsum[1]);
    f2_unpack(acc[1], lsum[2], lsum[3]);
  }
}

// WIN: a restricted-attention window is set (otherwise both sides are open at
// compile time, and the tile ranges reduce to the causal / padding ones).
template <int D, int NQ, int BN, bool WIN>
__global__ void __launch_bounds__(Fwd<D, NQ, BN>::THREADS, Fwd<D, NQ, BN>::MIN_BLOCKS)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const FwdParams p) {
  using C = Fwd<D, NQ, BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) FwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Causal: blocks in order of decreasing length (the longest query blocks of
  // every head first). Otherwise head-major (the launcher puts the query block
  // on x): the CTAs that run at the same time share few heads, so their K and
  // V stay in L2 instead of being read from HBM once per query block.
  const int bh = p.qb_fast ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x);
  const int y = p.qb_fast ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.y);
  const int qb = p.causal ? (p.num_qblocks - 1 - y) : y;
  const int q0 = qb * (NQ * 128);
  volatile int* abort_flag = &sh.abort_flag;
  const Watchdog wd = p.wd;
  const int wl = WIN ? p.wl : -1, wr = WIN ? p.wr : -1;

  // real keys of this head (key padding); per query tile g the key tiles
  // [jlo[g], jlo[g] + ntile[g]) that hold a key some row of the tile sees
  // (ntile 0 for tiles past n or without a visible key); the CTA loads the
  // union [jlo_cta, jlo_cta + nt) through its ring
  const int mb = head_keys(p.kv_len, bh, p.h, p.m);
  int ntile[NQ], jlo[NQ];
  int nt = 0, nq_valid = 0, jlo_cta = 0x7fffffff, jhi_cta = 0;
#pragma unroll
  for (int g = 0; g < NQ; ++g) {
    const int r0 = q0 + g * 128, r1 = min(r0 + 127, p.n - 1);
    int lo0, hi0, lo1, hi1;
    key_range(r0, mb, p.causal, wl, wr, lo0, hi0);  // row bounds are nondecreasing in the row
    key_range(r1, mb, p.causal, wl, wr, lo1, hi1);
    const bool any = r0 < p.n && hi1 > lo0;
    jlo[g] = any ? lo0 / BN : 0;
    ntile[g] = any ? (hi1 + BN - 1) / BN - jlo[g] : 0;
    if (ntile[g] > 0) {
      jlo_cta = min(jlo_cta, jlo[g]);
      jhi_cta = max(jhi_cta, jlo[g] + ntile[g]);
    }
    nq_valid += (r0 < p.n) ? 1 : 0;
  }
  if (jhi_cta > 0) nt = jhi_cta - jlo_cta;
  else jlo_cta = 0;

  if (tid == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      for (int g = 0; g < NQ; ++g) mbar_init(&sh.kv_empty[g][s], 1);
    }
    for (int g = 0; g < NQ; ++g) {
      mbar_init(&sh.s_full[g], 1);
      mbar_init(&sh.p_full[g], 128);
      mbar_init(&sh.o_full[g], 1);
      mbar_init(&sh.drain[g], 1);
      mbar_init(&sh.s_free[g], 128);
      mbar_init(&sh.pv_done[g], 1);
    }
    for (int g = 0; g < NQ; ++g) mbar_init(&sh.o_staged[g], 128);
    mbar_init(&sh.exp_turn[0], 128);
    mbar_init(&sh.exp_turn[1], 128);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::ISSUER) {
    tmem_alloc<C::TMEM_COLS>(&sh.tmem_base);
    tmem_relinquish();
  }
  if (warp == C::PRODUCER && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == C::PRODUCER) {
    // ------------------------------------------------------------ TMA producer
    if (C::REG_SPLIT) reg_dealloc<C::REG_OTHER>();
    if (lane == 0) {
      // bit s of `filled`: stage s was loaded; bit s of `last_ph`: parity of its last fill
      uint32_t filled = 0, last_ph = 0;
      mbar_arrive_expect_tx(&sh.q_full, nq_valid * C::QTILE);
      for (int t = 0; t < nq_valid; ++t)
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_Q + t * C::QTILE + a * C::QBOX, &tm_q, &sh.q_full, a * C::ATOM,
                      q0 + t * 128, bh);
      bool ok = true;
      for (int jj = 0; ok && jj < nt; ++jj) {
        // ring position jj holds key tile j; query tile g reads ring positions
        // [a, a + ntile[g]) with a = jlo[g] - jlo_cta
        const int j = jlo_cta + jj;
        const int st = jj % C::STAGES;
        const uint32_t ph = (jj / C::STAGES) & 1;
        // the stage's previous tile (ring position x = jj - STAGES) must be
        // released by every query tile that read it; it was that tile's use
        // number (x - a) / STAGES of the stage
        if (jj >= C::STAGES) {
          const int x = jj - C::STAGES;
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            const int a = jlo[g] - jlo_cta;
            if (ok && ntile[g] > 0 && x >= a && x < a + ntile[g])
              ok = guarded_wait(&sh.kv_empty[g][st], static_cast<uint32_t>((x - a) / C::STAGES) & 1u, abort_flag,
                                wd, kSiteKEmpty);
          }
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&sh.kv_full[st], 2 * C::KTILE);
        filled |= 1u << st;
        last_ph = (last_ph & ~(1u << st)) | (ph << st);
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_K + st * C::KTILE + a * C::KBOX, &tm_k, &sh.kv_full[st],
                      a * C::ATOM, j * BN, bh);
        if (p.inject == 1 && jj == 0) continue;  // test hook: this value tile never arrives
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_V + st * C::KTILE + a * C::KBOX, &tm_v, &sh.kv_full[st],
                      a * C::ATOM, j * BN, bh);
      }
      // Let every copy this thread started land before shared memory is released.
      drain_wait(&sh.q_full, 0, wd);
      for (int s = 0; s < C::STAGES; ++s)
        if ((filled >> s) & 1u) drain_wait(&sh.kv_full[s], (last_ph >> s) & 1u, wd);
    }
  } else if (warp >= C::ISSUER) {
    // ------------------------------------------------------------ MMA issuer of query tile g
    if (C::REG_SPLIT) reg_dealloc<C::REG_OTHER>();
    const int g = warp - C::ISSUER;
    int T = 0, a = 0;  // key tiles of this query tile, ring position of its first
#pragma unroll
    for (int gg = 0; gg < NQ; ++gg)
      if (gg == g) {
        T = ntile[gg];
        a = jlo[gg] - jlo_cta;
      }
    if (lane == 0 && T > 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, BN, false, false) | (p.neg ? (1u << 13) : 0u);
      const uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q) + g * C::QTILE;
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      const uint32_t t_s = tmem + C::tm_s(g), t_p = tmem + C::tm_p(g), t_o = tmem + C::tm_o(g);
      auto issue_s = [&](int st) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int a = k / (C::ATOM / 16), w = k % (C::ATOM / 16);
          const uint64_t da = smem_desc(sQ + a * C::QBOX + w * 32, 16, C::SBO, C::SWZ);
          const uint64_t db = smem_desc(sK + st * C::KTILE + a * C::KBOX + w * 32, 16, C::SBO, C::SWZ);
          mma_ss(t_s, da, db, idesc_s, k > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int st, bool acc) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t db = smem_desc(sV + st * C::KTILE + k * 16 * C::ATOM * 2, C::KBOX, C::SBO, C::SWZ);
          mma_ts(t_o, t_p + k * 8, db, idesc_o, (acc || k > 0) ? 1u : 0u);
        }
      };
      // this query tile's key tile j (0-based among its T) sits at ring position a + j
      bool ok = guarded_wait(&sh.q_full, 0, abort_flag, wd, kSiteQFull) &&
                guarded_wait(&sh.kv_full[a % C::STAGES], (a / C::STAGES) & 1, abort_flag, wd, kSiteKFull);
      if (ok) {
        issue_s(a % C::STAGES);
        mma_commit(&sh.s_full[g]);
      }
      for (int j = 0; ok && j < T; ++j) {
        const int st = (a + j) % C::STAGES;
        if (C::SEP_P && j + 1 < T) {
          // S_g(j+1) as soon as the softmax holds S_g(j) in registers
          const int jn = a + j + 1, stn = jn % C::STAGES;
          if (!(ok = guarded_wait(&sh.s_free[g], j & 1, abort_flag, wd, kSiteSFull))) break;
          if (!(ok = guarded_wait(&sh.kv_full[stn], (jn / C::STAGES) & 1, abort_flag, wd, kSiteKFull))) break;
          tc_fence_after();
          issue_s(stn);
          mma_commit(&sh.s_full[g]);
        }
        if (!(ok = guarded_wait(&sh.p_full[g], j & 1, abort_flag, wd, kSitePFull))) break;
        tc_fence_after();
        issue_pv(st, j > 0);
        if (C::SEP_P) mma_commit(&sh.pv_done[g]);
        if (j == T - 1) mma_commit(&sh.o_full[g]);
        mma_commit(&sh.kv_empty[g][st]);  // K_j and V_j are no longer read by this tile
        if (!C::SEP_P && j + 1 < T) {
          const int jn = a + j + 1, stn = jn % C::STAGES;
          if (!(ok = guarded_wait(&sh.kv_full[stn], (jn / C::STAGES) & 1, abort_flag, wd, kSiteKFull))) break;
          issue_s(stn);
          mma_commit(&sh.s_full[g]);
        }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit(&sh.drain[g]);
      drain_wait(&sh.drain[g], 0, wd);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups
    // Query tile g: the thread owns row r of the tile (TMEM lane r).
    if (C::REG_SPLIT) reg_alloc<C::REG_SOFTMAX>();
    const int g = warp / 4;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int row = q0 + g * 128 + r;
    int my_tiles = 0, my_jlo = 0;
#pragma unroll
    for (int gg = 0; gg < NQ; ++gg)
      if (gg == g) {
        my_tiles = ntile[gg];
        my_jlo = jlo[gg];
      }
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::tm_s(g);
    const uint32_t t_p = tmem + lane_base + C::tm_p(g);
    const uint32_t t_o = tmem + lane_base + C::tm_o(g);
    int klo, khi;  // visible keys [klo, khi) of this row
    key_range(row, mb, p.causal, wl, wr, klo, khi);
    // d <= 64: scale 0 runs with a tiny positive c (see the persistent kernel),
    // so one exponential loop serves masked and unmasked tiles (2-7 % faster for
    // the short and the causal shapes; at d = 128 the two loops measured faster)
    const float c = (D <= 64 && !(p.c > 0.f)) ? 1e-30f : p.c;
    const uint64_t c2 = f2_pack(c, c);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    // With two query tiles and P aliasing S, the exponentials of tile 0 and
    // tile 1 take turns (0, 1, 0, 1, ... per key tile), so that one group's
    // exponentials overlap the other group's MMAs instead of both groups
    // computing at once and then both waiting for the tensor cores. Group 0
    // waits for group 1's previous turn, group 1 for group 0's turn on the
    // same key tile, each only while the other group still has that tile.
    // (Both groups must start at the same key tile: not with a window.)
    constexpr bool turns = (NQ == 2) && !C::SEP_P && !WIN;
    int other_tiles = 0;
#pragma unroll
    for (int gg = 0; gg < NQ; ++gg)
      if (gg == (g ^ 1)) other_tiles = ntile[gg];
    if (turns && g == 1) mbar_arrive(&sh.exp_turn[0]);  // group 0 goes first
    for (int j = 0; j < my_tiles; ++j) {
      // a failed wait is acted on at the end of the iteration
      ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full[g], j & 1, abort_flag, wd, kSiteSFull)) && ok;
      tc_fence_after();
      uint32_t s[C::CHUNKS][32];
#pragma unroll
      for (int q = 0; q < C::CHUNKS; ++q) tmem_ld32(t_s + q * 32, s[q]);
      tmem_ld_wait();
      if (C::SEP_P) {
        tc_fence_before();
        mbar_arrive(&sh.s_free[g]);  // S_g may be overwritten by S_g(j+1)
      }
      // this row sees the tile's columns [rlo, rem) (key tile my_jlo + j)
      const int k0 = (my_jlo + j) * BN;
      const int rem = khi - k0, rlo = klo - k0;
      const bool masked = __any_sync(0xffffffffu, rem < C::COLS || rlo > 0);
      if (masked) {
#pragma unroll
        for (int q = 0; q < C::CHUNKS; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i >= rem || q * 32 + i < rlo) s[q][i] = __float_as_uint(-INFINITY);
      }
      // row max: four chains of 3-input max, seeded with columns 0..7; every
      // later step covers 8 columns, ending exactly at COLS
      float mx4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        mx4[u] = fmaxf(__uint_as_float(s[0][2 * u]), __uint_as_float(s[0][2 * u + 1]));
#pragma unroll
      for (int e = 8; e < C::COLS; e += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mx4[u] = max3(mx4[u], __uint_as_float(s[(e + 2 * u) >> 5][(e + 2 * u) & 31]),
                        __uint_as_float(s[(e + 2 * u + 1) >> 5][(e + 2 * u + 1) & 31]));
      }
      const float m_new = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m_used = m_new;
      } else if (m_new > m_used + kRescaleThreshold) {
        // (from -inf, a row whose window starts in this tile: alpha = 0, O and l are 0)
        alpha = ex2(m_used - m_new);
        m_used = m_new;
        rescale = true;
      }
      // a row with no visible key so far keeps the reference 0 (its weights are 0)
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
      if (turns && (g == 0 ? (j == 0 || j - 1 < other_tiles) : j < other_tiles))
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.exp_turn[g], j & 1, abort_flag, wd, kSiteExpTurn)) && ok;
      if (C::SEP_P && j > 0) {
        // PV_g(j-1) still reads P_g until it completes
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.pv_done[g], (j - 1) & 1, abort_flag, wd, kSitePFull)) && ok;
        tc_fence_after();
      }
      float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < C::CHUNKS; ++q) {
        uint32_t pk[16];
        // masked scores already hold -inf, and 2^(-inf * c - m) = 0 for c > 0;
        // only c = 0 (scale 0, d = 128) needs the explicit mask (-inf * 0 is NaN)
        if (D > 64 && masked && c == 0.f)
          exp_chunk<true, true>(s[q], q * 32, rlo, rem, c2, nm2, lsum, pk);
        else
          exp_chunk<false, true>(s[q], q * 32, rlo, rem, c2, nm2, lsum, pk);
        tmem_st16(t_p + q * 16, pk);
      }
      if (turns) mbar_arrive(&sh.exp_turn[g ^ 1]);  // the other group's turn
      l = l * alpha + ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3]));
      tmem_st_wait();
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        rescale_o<C::OCOLS>(t_o, alpha);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&sh.p_full[g]);
      if (!ok) break;
    }
    // a query tile without a visible key (a sequence without real keys, or a
    // window past the keys): its rows are the empty sum
    if (my_tiles == 0) write_empty_row<D>(p, bh, row, 0, D, true);
    if (ok && my_tiles > 0) {
      ok = __all_sync(0xffffffffu, guarded_wait(&sh.o_full[g], 0, abort_flag, wd, kSiteOFull));
      if (ok) {
        tc_fence_after();
        // a row that saw no key (l = 0) is the empty sum: O = 0, lse = -inf
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        // O leaves through the shared-memory tile of Q_g (no MMA reads it any
        // more once o_full completed), written in the TMA map's swizzled layout
        // and stored by one thread; rows past n are clipped by the map.
        uint8_t* qtile = smem + C::OFF_Q + g * C::QTILE;
#pragma unroll
        for (int q = 0; q < C::OCOLS / 16; ++q) {
          uint32_t o[16];
          tmem_ld16(t_o + q * 16, o);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = (q * 16) / 8 + u;                 // 16-byte chunk of the row
            constexpr int CPA = C::ATOM / 8;                 // chunks per swizzle atom row
            const int at = cc / CPA, ca = cc % CPA;
            const int pc = (C::ATOM == 64) ? (ca ^ (r & 7)) : (ca ^ ((r >> 1) & 3));
            *reinterpret_cast<uint4*>(qtile + at * C::QBOX + r * (C::ATOM * 2) + (pc << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sh.o_staged[g]);
        if (r == 0) {
          if (guarded_wait(&sh.o_staged[g], 0, abort_flag, wd, kSiteOFull)) {
            for (int at = 0; at < C::NATOM; ++at)
              tma_store_3d(&tm_o, qtile + at * C::QBOX, at * C::ATOM, q0 + g * 128, bh);
            tma_store_commit();
            tma_store_wait_all();  // before the CTA (and its shared memory) goes away
          }
        }
        if (row < p.n && p.lse != nullptr)
          p.lse[static_cast<size_t>(bh) * p.n + row] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::ISSUER) {
    tc_fence_after();
    tmem_dealloc<C::TMEM_COLS>(tmem);
  }
}

template <int D, int NQ, int BN, bool WIN>
cudaError_t launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, FwdParams p, int BH, cudaStream_t stream) {
  using C = Fwd<D, NQ, BN>;
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_fwd_kernel<D, NQ, BN, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  if (C::REG_SPLIT) {
    // setmaxnreg.inc waits until registers are free: the split must fit in the
    // registers the CTA is launched with, or the kernel would never proceed.
    static int regs_per_thread[64] = {0};
    if (regs_per_thread[dev & 63] == 0) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, attn_fwd_kernel<D, NQ, BN, WIN>)) != cudaSuccess) return e;
      regs_per_thread[dev & 63] = fa.numRegs;
    }
    if (regs_per_thread[dev & 63] * C::THREADS < C::SOFT_WARPS * 32 * C::REG_SOFTMAX + 128 * C::REG_OTHER)
      return cudaErrorInvalidConfiguration;
  }
  p.num_qblocks = (p.n + NQ * 128 - 1) / (NQ * 128);
  // grid y is limited to 65535: heads go on y only where they fit
  p.qb_fast = (!p.causal && BH <= 65535) ? 1 : 0;
  const dim3 grid = p.qb_fast ? dim3(static_cast<unsigned>(p.num_qblocks), static_cast<unsigned>(BH))
                              : dim3(static_cast<unsigned>(BH), static_cast<unsigned>(p.num_qblocks));
  prof_begin(kKindFwd, stream);
  attn_fwd_kernel<D, NQ, BN, WIN><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, to, p);
  e = cudaGetLastError();
  prof_end(kKindFwd, stream);
  return e;
}

// ---------------------------------------------------------------- persistent forward (d <= 64)
//
// One CTA per SM loops over work items (head, 256 query rows); items are
// taken in launch order (causal: the blocks with the most key tiles first).
// The two query tiles of an item are handled as in attn_fwd_kernel with P in
// TMEM columns of its own. Across items: Q in two sets (the next item's Q
// loads while the current one runs), one continuous K/V ring, and each query
// tile's O epilogue (TMEM -> shared memory -> TMA store) overlaps the next
// item's first score product, which only needs S to be free. The next item's
// first P.V product waits until the epilogue has read O out of TMEM.
// TMEM: S_0 S_1 [0,256), P_0 P_1 [256,384) (bf16 pairs), O_0 O_1 [384,384+2D).
//
// Items of at most two key tiles (SHORT: m <= 256) are short enough that the
// item boundary sets their rate. There the next item's first score product is
// issued as soon as the softmax holds this item's last scores, the softmax
// takes the next item's first exponentials before this item's epilogue (so
// the last P.V runs under them), and O leaves through a staging tile of its
// own, so the issuers release an item's Q set once its last score product has
// read it (four K/V stages make room for the staging tiles).
template <int D, bool SHORT = false>
struct FwdP {
  static constexpr int NQ = 2, BN = 128;
  static constexpr int ATOM = D;                          // one swizzle atom per row (D <= 64)
  static constexpr uint32_t SWZ = (D == 64) ? 2u : 4u;
  static constexpr uint32_t SBO = 8u * ATOM * 2u;
  static constexpr uint32_t QTILE = 128u * D * 2u;
  static constexpr uint32_t KTILE = BN * D * 2u;
  // K/V ring depth: a tile takes about 2.5 us from its TMA issue to its
  // arrival when every SM streams keys (measured with a clock64 trace at
  // n = m = 16384, d = 64), more than four stages of about 1.2 us cover
  static constexpr int STAGES = SHORT ? 4 : 5;
  static constexpr uint32_t OFF_Q = 0;                    // 2 sets x NQ tiles
  static constexpr uint32_t OFF_K = 2 * NQ * QTILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KTILE;
  static constexpr uint32_t OFF_OSTG = OFF_V + STAGES * KTILE;  // SHORT: O staging, one tile per query tile
  static constexpr uint32_t SMEM = OFF_OSTG + (SHORT ? NQ * QTILE : 0u) + 1024;
  static constexpr int THREADS = NQ * 128 + 128;          // softmax, producer, issuers, idle
  static constexpr int PRODUCER = 4 * NQ, ISSUER = 4 * NQ + 1;
  // setmaxnreg split of the 384 x 168 registers the CTA is launched with: the
  // softmax keeps a tile's scores and its packed weights in registers at once
  static constexpr int REG_SOFTMAX = 224, REG_OTHER = 56;
  static_assert(NQ * 128 * REG_SOFTMAX + 128 * REG_OTHER <= 384 * 168, "register split");
  static_assert(SMEM + sizeof(uint64_t) * 64 <= 227u * 1024u, "shared memory per block");
  static constexpr int CHUNKS = BN / 32;
  static constexpr uint32_t P_COLS = BN / 2;
  __host__ __device__ static constexpr uint32_t tm_s(int g) { return g * BN; }
  __host__ __device__ static constexpr uint32_t tm_p(int g) { return NQ * BN + g * P_COLS; }
  __host__ __device__ static constexpr uint32_t tm_o(int g) { return NQ * (BN + P_COLS) + g * D; }
  static_assert(NQ * (BN + P_COLS + D) <= 512, "TMEM columns");
};

struct FwdPShared {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[2][kMaxStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_full[2], o_free[2], o_staged[2];
  uint64_t ostg_free[2];  // SHORT: the O store of the staging tile has read it
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, bool SPEC>
__global__ void __launch_bounds__(FwdP<D, !SPEC>::THREADS, 1)
attn_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const FwdParams p, int BH, int items) {
  using C = FwdP<D, !SPEC>;
  constexpr bool SHORT = !SPEC;
  constexpr int NQ = C::NQ, BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) FwdPShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const Watchdog wd = p.wd;
  // item -> (head, first query row); key tiles per query tile (0 past n)
  // item -> (head, first query row, real keys of the head)
  auto item_of = [&](int it, int& bh, int& q0, int& mb, int (&ntile)[2], int& nt, int& nq_valid) {
    // causal: the longest query blocks of every head first; otherwise head-major
    // (CTAs working at the same time share the heads' K and V in L2)
    bh = p.causal ? it % BH : it / p.num_qblocks;
    const int y = p.causal ? it / BH : it % p.num_qblocks;
    const int qb = p.causal ? (p.num_qblocks - 1 - y) : y;
    q0 = qb * (NQ * 128);
    mb = head_keys(p.kv_len, bh, p.h, p.m);
    nt = 0;
    nq_valid = 0;
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
      const int r0 = q0 + g * 128;
      ntile[g] = (r0 < p.n && mb > 0) ? key_tiles<BN>(min(r0 + 127, p.n - 1), mb, p.causal) : 0;
      nt = max(nt, ntile[g]);
      nq_valid += (r0 < p.n) ? 1 : 0;
    }
  };

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.q_empty[s], NQ);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      for (int g = 0; g < NQ; ++g) mbar_init(&sh.kv_empty[g][s], 1);
    }
    for (int g = 0; g < NQ; ++g) {
      mbar_init(&sh.s_full[g], 1);
      mbar_init(&sh.s_free[g], 128);
      mbar_init(&sh.p_full[g], 128);
      mbar_init(&sh.pv_done[g], 1);
      mbar_init(&sh.o_full[g], 1);
      mbar_init(&sh.o_free[g], 128);
      mbar_init(&sh.o_staged[g], 128);
      mbar_init(&sh.ostg_free[g], 1);
      mbar_init(&sh.drain[g], 1);
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::ISSUER) {
    tmem_alloc<512>(&sh.tmem_base);
    tmem_relinquish();
  }
  if (warp == C::PRODUCER && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == C::PRODUCER) {
    // ------------------------------------------------------------ TMA producer
    if constexpr (SPEC) reg_dealloc<C::REG_OTHER>();
    if (lane == 0) {
      // per stage s, group g (bit g * 8 + s): `users` = the stage's last tile was
      // used by group g; `uses` = parity of group g's uses of stage s so far
      uint32_t users = 0, uses = 0, kv_filled = 0, kv_ph = 0, q_filled = 0, q_ph = 0;
      int jj = 0;
      bool ok = true;
      for (int it = blockIdx.x, li = 0; ok && it < items; it += gridDim.x, ++li) {
        int bh, q0, mb, ntile[2], nt, nq_valid;
        item_of(it, bh, q0, mb, ntile, nt, nq_valid);
        const int qs = li & 1;
        if (li >= 2 && !(ok = guarded_wait(&sh.q_empty[qs], ((li >> 1) - 1) & 1, abort_flag, wd, kSiteKEmpty)))
          break;
        if (nt > 0) {
          mbar_arrive_expect_tx(&sh.q_full[qs], nq_valid * C::QTILE);
          for (int t = 0; t < nq_valid; ++t)
            tma_load_3d(smem + C::OFF_Q + (qs * NQ + t) * C::QTILE, &tm_q, &sh.q_full[qs], 0, q0 + t * 128, bh);
        } else {
          // no key tile (a sequence without real keys): no MMA reads Q, so none
          // is loaded, but the set's phase still completes
          mbar_arrive(&sh.q_full[qs]);
        }
        q_filled |= 1u << qs;
        q_ph = (q_ph & ~(1u << qs)) | (static_cast<uint32_t>((li >> 1) & 1) << qs);
        for (int j = 0; ok && j < nt; ++j, ++jj) {
          const int st = jj % C::STAGES;
          // the stage's previous tile must be released by every query tile that used it
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            const uint32_t bit = 1u << (g * 8 + st);
            if (ok && (users & bit))
              ok = guarded_wait(&sh.kv_empty[g][st], ((uses & bit) ? 1u : 0u) ^ 1u, abort_flag, wd, kSiteKEmpty);
          }
          if (!ok) break;
          mbar_arrive_expect_tx(&sh.kv_full[st], 2 * C::KTILE);
          kv_filled |= 1u << st;
          kv_ph = (kv_ph & ~(1u << st)) | (static_cast<uint32_t>((jj / C::STAGES) & 1) << st);
          tma_load_3d(smem + C::OFF_K + st * C::KTILE, &tm_k, &sh.kv_full[st], 0, j * BN, bh);
          if (!(p.inject == 1 && jj == 0))  // test hook: this value tile never arrives
            tma_load_3d(smem + C::OFF_V + st * C::KTILE, &tm_v, &sh.kv_full[st], 0, j * BN, bh);
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            const uint32_t bit = 1u << (g * 8 + st);
            if (j < ntile[g]) {
              users |= bit;
              uses ^= bit;
            } else {
              users &= ~bit;
            }
          }
        }
      }
      // Let every copy this thread started land before shared memory is released.
      for (int s = 0; s < 2; ++s)
        if ((q_filled >> s) & 1u) drain_wait(&sh.q_full[s], (q_ph >> s) & 1u, wd);
      for (int s = 0; s < C::STAGES; ++s)
        if ((kv_filled >> s) & 1u) drain_wait(&sh.kv_full[s], (kv_ph >> s) & 1u, wd);
    }
  } else if (warp >= C::ISSUER) {
    // ------------------------------------------------------------ MMA issuer of query tile g
    if constexpr (SPEC) reg_dealloc<C::REG_OTHER>();
    const int g = warp - C::ISSUER;
    if (lane == 0 && g < NQ) {
      const uint32_t idesc_s = idesc_bf16_f32(128, BN, false, false) | (p.neg ? (1u << 13) : 0u);
      const uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      const uint32_t t_s = tmem + C::tm_s(g), t_p = tmem + C::tm_p(g), t_o = tmem + C::tm_o(g);
      auto issue_s = [&](uint32_t sQ, int st) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t da = smem_desc(sQ + k * 32, 16, C::SBO, C::SWZ);
          const uint64_t db = smem_desc(sK + st * C::KTILE + k * 32, 16, C::SBO, C::SWZ);
          mma_ss(t_s, da, db, idesc_s, k > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int st, bool acc) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t db = smem_desc(sV + st * C::KTILE + k * 16 * C::ATOM * 2, C::KTILE, C::SBO, C::SWZ);
          mma_ts(t_o, t_p + k * 8, db, idesc_o, (acc || k > 0) ? 1u : 0u);
        }
      };
      bool ok = true;
      int jj = 0, gt = 0, oc = 0;  // K/V tiles of earlier items, this tile's S count, items with output
      bool s0_ahead = false;       // SHORT: this item's first S was issued during the previous item
      for (int it = blockIdx.x, li = 0; ok && it < items; it += gridDim.x, ++li) {
        int bh, q0, mb, ntile[2], nt, nq_valid;
        item_of(it, bh, q0, mb, ntile, nt, nq_valid);
        const int T = g == 0 ? ntile[0] : ntile[1];
        if (T > 0) {
          const uint32_t sQ = smem_u32(smem + C::OFF_Q) + ((li & 1) * NQ + g) * C::QTILE;
          if (!s0_ahead) {
            // S of this item's first tile: Q landed, K_0 landed, the softmax holds the previous S
            ok = guarded_wait(&sh.q_full[li & 1], (li >> 1) & 1, abort_flag, wd, kSiteQFull) &&
                 guarded_wait(&sh.kv_full[jj % C::STAGES], (jj / C::STAGES) & 1, abort_flag, wd, kSiteKFull) &&
                 (gt == 0 || guarded_wait(&sh.s_free[g], (gt - 1) & 1, abort_flag, wd, kSiteSFull));
            if (!ok) break;
            tc_fence_after();
            issue_s(sQ, jj % C::STAGES);
            mma_commit(&sh.s_full[g]);
          }
          s0_ahead = false;
          // SHORT: the Q set is released to the producer once this item's last S read it
          if (SHORT && T == 1) mma_commit(&sh.q_empty[li & 1]);
          for (int j = 0; ok && j < T; ++j) {
            const int st = (jj + j) % C::STAGES;
            if (j + 1 < T) {
              const int jn = jj + j + 1;
              if (!(ok = guarded_wait(&sh.s_free[g], (gt + j) & 1, abort_flag, wd, kSiteSFull))) break;
              if (!(ok = guarded_wait(&sh.kv_full[jn % C::STAGES], (jn / C::STAGES) & 1, abort_flag, wd, kSiteKFull)))
                break;
              tc_fence_after();
              issue_s(sQ, jn % C::STAGES);
              mma_commit(&sh.s_full[g]);
              if (SHORT && j + 2 == T) mma_commit(&sh.q_empty[li & 1]);
            } else if (SHORT && it + static_cast<int>(gridDim.x) < items) {
              // the next item's first S, ahead of this item's last P.V
              int bh2, q02, mb2, ntile2[2], nt2, nq2;
              item_of(it + gridDim.x, bh2, q02, mb2, ntile2, nt2, nq2);
              if ((g == 0 ? ntile2[0] : ntile2[1]) > 0) {
                const int l2 = li + 1, jn = jj + nt;
                ok = guarded_wait(&sh.s_free[g], (gt + j) & 1, abort_flag, wd, kSiteSFull) &&
                     guarded_wait(&sh.q_full[l2 & 1], (l2 >> 1) & 1, abort_flag, wd, kSiteQFull) &&
                     guarded_wait(&sh.kv_full[jn % C::STAGES], (jn / C::STAGES) & 1, abort_flag, wd, kSiteKFull);
                if (!ok) break;
                tc_fence_after();
                issue_s(smem_u32(smem + C::OFF_Q) + ((l2 & 1) * NQ + g) * C::QTILE, jn % C::STAGES);
                mma_commit(&sh.s_full[g]);
                s0_ahead = true;
              }
            }
            if (!(ok = guarded_wait(&sh.p_full[g], (gt + j) & 1, abort_flag, wd, kSitePFull))) break;
            // the first P.V of an item overwrites O: the previous item's epilogue must have read it
            if (j == 0 && oc >= 1 && !(ok = guarded_wait(&sh.o_free[g], (oc - 1) & 1, abort_flag, wd, kSiteOFull)))
              break;
            tc_fence_after();
            issue_pv(st, j > 0);
            mma_commit(&sh.pv_done[g]);
            if (j == T - 1) mma_commit(&sh.o_full[g]);
            mma_commit(&sh.kv_empty[g][st]);  // K and V of this tile are no longer read by this query tile
          }
          gt += T;
          ++oc;
        } else if (SHORT) {
          mbar_arrive(&sh.q_empty[li & 1]);  // no S of this query tile reads the set
        }
        jj += nt;
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit(&sh.drain[g]);
      drain_wait(&sh.drain[g], 0, wd);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax of query tile g
    if constexpr (SPEC) reg_alloc<C::REG_SOFTMAX>();
    const int g = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::tm_s(g);
    const uint32_t t_p = tmem + lane_base + C::tm_p(g);
    const uint32_t t_o = tmem + lane_base + C::tm_o(g);
    // Scale 0 runs with a tiny positive c instead of 0: every score times c is
    // then far below the fp32 spacing at the reference, so each visible weight
    // is exactly 1 as for c = 0, while the masked scores (-inf) keep weight 0
    // (-inf * 0 would be NaN) without a second, masking copy of the exp loop
    // (the smaller loop measured 2 % faster at n = m = 16384, d = 64).
    const float c = p.c > 0.f ? p.c : 1e-30f;
    const uint64_t c2 = f2_pack(c, c);
    bool ok = true;
    int gt = 0, oc = 0;
    // Q set (SHORT: the staging tile, 0) whose O store thread 0 issued but has
    // not yet seen read (-1: none). The wait for the store is deferred to the
    // next item so that thread 0 (and with it the group) is not held up by the
    // store's latency.
    int pending_q = -1;
    auto release_pending = [&]() {
      if (r == 0 && pending_q >= 0) {
        bulk_wait_read_all();
        if (SHORT)
          mbar_arrive(&sh.ostg_free[g]);  // the staging tile may take the next item's O
        else
          mbar_arrive(&sh.q_empty[pending_q]);  // this Q tile may take a later item's rows
        pending_q = -1;
      }
    };
    // An item's epilogue: O / l into its Q tile (no MMA reads it once o_full
    // completed), one thread stores it (rows past n are clipped by the map), lse.
    // (Deferring it past the next item's first key tile measured slower for
    // short items: that item's Q then loads later.)
    struct ItemOut {
      int qs, q0, bh, row, oc;
      float l, m;
    };
    auto epilogue = [&](const ItemOut& ep) -> bool {
      if (!__all_sync(0xffffffffu, guarded_wait(&sh.o_full[g], ep.oc & 1, abort_flag, wd, kSiteOFull))) return false;
      tc_fence_after();
      const float inv_l = 1.f / ep.l;
      uint32_t w[D / 2];
#pragma unroll
      for (int q = 0; q < D / 16; ++q) {
        uint32_t o[16];
        tmem_ld16(t_o + q * 16, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[q * 8 + i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
      }
      tc_fence_before();
      mbar_arrive(&sh.o_free[g]);  // the next item's first P.V may overwrite O
      uint8_t* qtile = SHORT ? smem + C::OFF_OSTG + g * C::QTILE : smem + C::OFF_Q + (ep.qs * NQ + g) * C::QTILE;
      if (SHORT && ep.oc >= 1) {
        // the previous item's store must have read the staging tile
        release_pending();
        if (!__all_sync(0xffffffffu, guarded_wait(&sh.ostg_free[g], (ep.oc - 1) & 1, abort_flag, wd, kSiteOFull)))
          return false;
      }
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        const int pc = (D == 64) ? (ch ^ (r & 7)) : (ch ^ ((r >> 1) & 3));
        *reinterpret_cast<uint4*>(qtile + r * (D * 2) + (pc << 4)) =
            make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh.o_staged[g]);
      if (r == 0) {
        release_pending();  // the previous item's store, long done by now
        if (guarded_wait(&sh.o_staged[g], ep.oc & 1, abort_flag, wd, kSiteOFull)) {
          tma_store_3d(&tm_o, qtile, 0, ep.q0 + g * 128, ep.bh);
          tma_store_commit();
        }
        pending_q = ep.qs;
      }
      if (ep.row < p.n && p.lse != nullptr)
        p.lse[static_cast<size_t>(ep.bh) * p.n + ep.row] = (ep.m + log2f(ep.l)) * kLn2;
      return true;
    };
    // SHORT: the previous item's epilogue, taken after this item's first exponentials
    bool have_ep = false;
    ItemOut pend{};
    for (int it = blockIdx.x, li = 0; ok && it < items; it += gridDim.x, ++li) {
      int bh, q0, mb, ntile[2], nt, nq_valid;
      item_of(it, bh, q0, mb, ntile, nt, nq_valid);
      const int T = g == 0 ? ntile[0] : ntile[1];
      const int qs = li & 1;
      if (T == 0) {
        if (mb == 0) write_empty_row<D>(p, bh, q0 + g * 128 + r, 0, D, true);
        if (SHORT) {
          // the previous item's deferred epilogue (SHORT) is written before anything else
          if (have_ep && !(ok = epilogue(pend))) break;
          have_ep = false;
          continue;
        }
        release_pending();
        // no rows of this item here: the Q set does not wait for this tile's output
        if (r == 0) mbar_arrive(&sh.q_empty[qs]);
        continue;
      }
      const int row = q0 + g * 128 + r;
      const int lim = p.causal ? min(row + 1, mb) : mb;  // keys [0, lim) are visible
      float m_used = 0.f, l = 0.f;
      if constexpr (SPEC) {
        for (int j = 0; j < T; ++j) {
          const int gj = gt + j;
          ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full[g], gj & 1, abort_flag, wd, kSiteSFull));
          if (!ok) break;
          tc_fence_after();
          if (j <= 1) release_pending();  // (a no-op at j = 1; this placement measured faster)
          uint32_t s[C::CHUNKS][32];
  #pragma unroll
          for (int q = 0; q < C::CHUNKS; ++q) tmem_ld32(t_s + q * 32, s[q]);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&sh.s_free[g]);  // S may be overwritten by the next score product
          const int rem = lim - j * BN;
          const bool masked = __any_sync(0xffffffffu, rem < BN);
          if (masked) {
  #pragma unroll
            for (int q = 0; q < C::CHUNKS; ++q)
  #pragma unroll
              for (int i = 0; i < 32; ++i)
                if (q * 32 + i >= rem) s[q][i] = __float_as_uint(-INFINITY);
          }
          // Row maximum of the tile (scaled, log2 units).
          auto tile_max = [&]() {
            float mx4[4];
  #pragma unroll
            for (int u = 0; u < 4; ++u)
              mx4[u] = fmaxf(__uint_as_float(s[0][2 * u]), __uint_as_float(s[0][2 * u + 1]));
  #pragma unroll
            for (int e = 8; e < BN; e += 8) {
  #pragma unroll
              for (int u = 0; u < 4; ++u)
                mx4[u] = max3(mx4[u], __uint_as_float(s[(e + 2 * u) >> 5][(e + 2 * u) & 31]),
                              __uint_as_float(s[(e + 2 * u + 1) >> 5][(e + 2 * u + 1) & 31]));
            }
            return fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
          };
          // The first two tiles of an item take their row maximum (lazy rescale
          // as in attn_fwd_kernel). From the third tile on, a tile is
          // exponentiated against the running reference without a maximum pass;
          // a tile sum above kSpecLimitSum shows that the scores grew, and only
          // then is the tile's maximum taken and the row moved to it.
          const bool spec = j >= 2;
          float alpha = 1.f;
          bool rescale = false;
          if (!spec) {
            const float m_new = tile_max();
            if (j == 0) {
              m_used = m_new;
            } else if (m_new > m_used + kRescaleThreshold) {
              alpha = ex2(m_used - m_new);
              m_used = m_new;
              rescale = true;
            }
          }
          uint32_t pk[C::CHUNKS][16];
          float lsum[4];
          // weights of the tile against m_used into pk; returns their sum
          auto exps = [&]() {
            const uint64_t nm2 = f2_pack(-m_used, -m_used);
            lsum[0] = lsum[1] = lsum[2] = lsum[3] = 0.f;
  #pragma unroll
            for (int q = 0; q < C::CHUNKS; ++q) exp_chunk<false, false>(s[q], 0, 0, 0, c2, nm2, lsum, pk[q]);
            return (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
          };
          // the weights are computed while the previous P.V still runs, then stored
          float l_tile = exps();
          bool pv_waited = false;
          if (spec) {
            const bool grew = !(l_tile <= kSpecLimitSum);  // also catches inf / NaN
            if (__any_sync(0xffffffffu, grew)) {
              if (grew) {
                const float m_new = tile_max();
                alpha = ex2(m_used - m_new);
                m_used = m_new;
              }
              l_tile = exps();  // unchanged for the rows that did not grow
              // O follows the moved reference (alpha = 1 for the other rows) once
              // the previous P.V has added to it, before this tile's P.V does; the
              // vote above is the only one the speculative tiles take for this
              ok = __all_sync(0xffffffffu, guarded_wait(&sh.pv_done[g], (gj - 1) & 1, abort_flag, wd, kSitePFull));
              if (!ok) break;
              tc_fence_after();
              pv_waited = true;
              rescale_o<D>(t_o, alpha);
            }
          }
          if (gj >= 1 && !pv_waited) {
            // the previous P.V (possibly the previous item's) still reads P until it completes
            ok = __all_sync(0xffffffffu, guarded_wait(&sh.pv_done[g], (gj - 1) & 1, abort_flag, wd, kSitePFull));
            if (!ok) break;
            tc_fence_after();
          }
  #pragma unroll
          for (int q = 0; q < C::CHUNKS; ++q) tmem_st16(t_p + q * 16, pk[q]);
          l = l * alpha + l_tile;
          if (!spec && j > 0 && __any_sync(0xffffffffu, rescale)) rescale_o<D>(t_o, alpha);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sh.p_full[g]);
        }
      } else {
        // SHORT items (at most two key tiles): every tile takes its maximum
        for (int j = 0; j < T; ++j) {
          const int gj = gt + j;
          ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full[g], gj & 1, abort_flag, wd, kSiteSFull));
          if (!ok) break;
          tc_fence_after();
          if (j <= 1) release_pending();  // (a no-op at j = 1)
          uint32_t s[C::CHUNKS][32];
  #pragma unroll
          for (int q = 0; q < C::CHUNKS; ++q) tmem_ld32(t_s + q * 32, s[q]);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&sh.s_free[g]);  // S may be overwritten by the next score product
          const int rem = lim - j * BN;
          const bool masked = __any_sync(0xffffffffu, rem < BN);
          if (masked) {
  #pragma unroll
            for (int q = 0; q < C::CHUNKS; ++q)
  #pragma unroll
              for (int i = 0; i < 32; ++i)
                if (q * 32 + i >= rem) s[q][i] = __float_as_uint(-INFINITY);
          }
          float mx4[4];
  #pragma unroll
          for (int u = 0; u < 4; ++u)
            mx4[u] = fmaxf(__uint_as_float(s[0][2 * u]), __uint_as_float(s[0][2 * u + 1]));
  #pragma unroll
          for (int e = 8; e < BN; e += 8) {
  #pragma unroll
            for (int u = 0; u < 4; ++u)
              mx4[u] = max3(mx4[u], __uint_as_float(s[(e + 2 * u) >> 5][(e + 2 * u) & 31]),
                            __uint_as_float(s[(e + 2 * u + 1) >> 5][(e + 2 * u + 1) & 31]));
          }
          const float m_new = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
          float alpha = 1.f;
          bool rescale = false;
          if (j == 0) {
            m_used = m_new;
          } else if (m_new > m_used + kRescaleThreshold) {
            alpha = ex2(m_used - m_new);
            m_used = m_new;
            rescale = true;
          }
          const uint64_t nm2 = f2_pack(-m_used, -m_used);
          // the weights stay in registers while the previous P.V (the previous
          // item's last one at j = 0) finishes and the previous item's O leaves
          float lsum[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[C::CHUNKS][16];
  #pragma unroll
          for (int q = 0; q < C::CHUNKS; ++q) exp_chunk<false, true>(s[q], 0, 0, 0, c2, nm2, lsum, pk[q]);
          if (j == 0 && have_ep) {
            have_ep = false;
            if (!(ok = epilogue(pend))) break;
          }
          if (gj >= 1) {
            // the previous P.V (possibly the previous item's) still reads P until it completes
            ok = __all_sync(0xffffffffu, guarded_wait(&sh.pv_done[g], (gj - 1) & 1, abort_flag, wd, kSitePFull));
            if (!ok) break;
            tc_fence_after();
          }
  #pragma unroll
          for (int q = 0; q < C::CHUNKS; ++q) tmem_st16(t_p + q * 16, pk[q]);
          l = l * alpha + ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3]));
          tmem_st_wait();
          if (j > 0 && __any_sync(0xffffffffu, rescale)) {
            rescale_o<D>(t_o, alpha);
            tmem_st_wait();
          }
          tc_fence_before();
          mbar_arrive(&sh.p_full[g]);
        }
      }
      if (!ok) break;
      if (SHORT) {
        pend = ItemOut{qs, q0, bh, row, oc, l, m_used};
        have_ep = true;
      } else {
        release_pending();
        if (!(ok = epilogue(ItemOut{qs, q0, bh, row, oc, l, m_used}))) break;
      }
      gt += T;
      ++oc;
    }
    if (SHORT && ok && have_ep) ok = epilogue(pend);
    release_pending();
    if (r == 0) tma_store_wait_all();  // stores must complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::ISSUER) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int D, bool SPEC>
cudaError_t launch_fwd_persist_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& to, FwdParams p, int BH, cudaStream_t stream) {
  using C = FwdP<D, !SPEC>;
  static std::once_flag once[64];
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_fwd_persist_kernel<D, SPEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  if (sm_count[dev & 63] == 0) {
    if (SPEC) {
      // setmaxnreg.inc waits until registers are free: the split must fit in the
      // registers the CTA is launched with, or the kernel would never proceed.
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, attn_fwd_persist_kernel<D, SPEC>)) != cudaSuccess) return e;
      if (fa.numRegs * C::THREADS < C::NQ * 128 * C::REG_SOFTMAX + 128 * C::REG_OTHER)
        return cudaErrorInvalidConfiguration;
    }
    int c = 0;
    if ((e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    sm_count[dev & 63] = c > 0 ? c : 1;
  }
  p.num_qblocks = (p.n + C::NQ * 128 - 1) / (C::NQ * 128);
  const long long items_ll = static_cast<long long>(BH) * p.num_qblocks;
  if (items_ll > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int items = static_cast<int>(items_ll);
  const int grid = items < sm_count[dev & 63] ? items : sm_count[dev & 63];
  prof_begin(kKindFwd, stream);
  attn_fwd_persist_kernel<D, SPEC><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, to, p, BH, items);
  e = cudaGetLastError();
  prof_end(kKindFwd, stream);
  return e;
}

// Speculative exponentials pay off from the third key tile of an item on;
// with at most two (m <= 256) every tile takes its maximum and no register
// split is needed.
template <int D>
cudaError_t launch_fwd_persist(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& to, const FwdParams& p, int BH, cudaStream_t stream) {
  if (p.m > 2 * FwdP<D>::BN) return launch_fwd_persist_cfg<D, true>(tq, tk, tv, to, p, BH, stream);
  return launch_fwd_persist_cfg<D, false>(tq, tk, tv, to, p, BH, stream);
}

}  // namespace

// Which forward kernel runs (measured on GB300, see the launcher below).
namespace {
// The persistent kernel handles neither the causal mask nor a window (the
// per-item kernel skips their masked key tiles per query tile).
bool fwd_persistent(int d, int n, int m, int causal, bool windowed) {
  // Causal: only very long query sequences, whose items differ most in length
  // (the persistent kernel takes the longest first). n = m = 16384, d = 64:
  // 2316 us against 2445 for the per-item kernel; n = 4096 equal, n = 1024 9 %
  // slower, short sequences slower still.
  if (causal) return d <= 64 && !windowed && n >= 8192 && (m % 128 == 0 || m >= 1024);
  return d <= 64 && !windowed && (m % 128 == 0 || m >= 1024);
}
}  // namespace

int fwd_key_tile(int d, int n, int m, int causal, bool windowed) {
  if (fwd_persistent(d, n, m, causal, windowed)) return 128;
  return (d >= 128 || n > 256) ? 128 : 64;
}

// Configuration: two 128-row query tiles per item. Non-causal d <= 64 with
// whole 128-key tiles (or long key sequences), and causal d <= 64 from 8192
// query rows on: the persistent kernel (P in TMEM columns of its own, items
// overlapped). Otherwise one CTA per item:
// 128-key tiles, or for d <= 64 with n <= 256 64-key tiles that halve TMEM to
// 256 columns so two CTAs share an SM (ragged or causal short sequences
// measured faster this way).
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, int BH, cudaStream_t stream) {
  const bool windowed = p.wl >= 0 || p.wr >= 0;
  const bool persist = fwd_persistent(d, p.n, p.m, p.causal, windowed);
  const bool small_tiles = fwd_key_tile(d, p.n, p.m, p.causal, windowed) == 64;
#define ATTN_FWD_CFG(D_, BN_)                                                  \
  (windowed ? launch_fwd_cfg<D_, 2, BN_, true>(tq, tk, tv, to, p, BH, stream) \
            : launch_fwd_cfg<D_, 2, BN_, false>(tq, tk, tv, to, p, BH, stream))
  switch (d) {
    case 32:
      if (persist) return launch_fwd_persist<32>(tq, tk, tv, to, p, BH, stream);
      return small_tiles ? ATTN_FWD_CFG(32, 64) : ATTN_FWD_CFG(32, 128);
    case 64:
      if (persist) return launch_fwd_persist<64>(tq, tk, tv, to, p, BH, stream);
      return small_tiles ? ATTN_FWD_CFG(64, 64) : ATTN_FWD_CFG(64, 128);
    case 128: return ATTN_FWD_CFG(128, 128);
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_FWD_CFG
}

}  // namespace attn
