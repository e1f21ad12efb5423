// Backward for short query sequences: one CTA owns whole heads.
//
// Same derivative as the general backward (attn_bwd.cu; "Attention Is All
// You Need", §3.2.1 eq. (1), differentiated):
//   P_ij = exp(scale q_i.k_j - lse_i),  D_i = sum_c dO_ic O_ic,
//   dS_ij = P_ij (dO_i . v_j - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
//
// When a head has at most two 128-row query tiles (n <= 256) and d <= 64, the
// fp32 dQ of every query row of the head fits in TMEM next to the other
// accumulators. A CTA then loops over all key tiles of a head, keeps dQ in
// TMEM across them, and writes bf16 dQ once at the end of the head: no fp32
// accumulator in global memory, no reduce-adds, no separate pre and post
// passes (D_i and lse_i * log2(e) are computed in the kernel). One launch,
// persistent CTAs over the heads.
//
// Per (key tile j, query tile i) the five products of the general kernel:
//   S^T = K_j Q_i^T, dP^T = V_j dO_i^T              (TMEM, lanes = keys)
//   dV_j += P^T dO_i   (P^T bf16 in TMEM, aliasing S^T)
//   dK_j += dS^T Q_i   (dS^T bf16 in shared memory, K-major view)
//   dQ_i += dS K_j     (same buffer, MN-major view; dQ_i stays in TMEM)
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D),
// dQ_i [256+2D+i*D, 256+2D+(i+1)*D).
//
// Shared memory: K/V in two sets (the next key tile loads during the current
// one), Q/dO tiles in a ring of three slots (a head holds one slot per query
// tile for all its key tiles; the third slot takes the next head's first
// tile early), per slot the rows' lse*log2(e) and D, and the dS^T tile.
//
// Warps (512 threads): 0-3 and 4-7 one thread per key row on query columns
// 0..63 / 64..127 (P, dS, dK/dV epilogue); 8-11 one thread per query row for
// the dQ epilogue; 12 TMA producer; 13 MMA issuer; 14-15 the per-row
// statistics D_i and lse_i * log2(e) of each arriving query tile.
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr float kLog2eH = 1.4426950408889634074f;

template <int D>
struct BwdHead {
  static_assert(D == 32 || D == 64, "whole-head backward: d <= 64");
  static constexpr int ATOM = D;                          // one swizzle atom per row
  static constexpr uint32_t SWZ = (D == 64) ? 2u : 4u;    // 128B / 64B swizzle
  static constexpr uint32_t SBO = 8u * ATOM * 2u;
  static constexpr uint32_t TILE = 128u * D * 2u;
  static constexpr uint32_t DS_REGION = 128u * 64u * 2u;
  static constexpr int NSLOT = 3;                         // Q/dO ring
  static constexpr int MAX_QT = 2;                        // query tiles per head
  static constexpr uint32_t OFF_K = 0;                    // 2 sets
  static constexpr uint32_t OFF_V = 2 * TILE;             // 2 sets
  static constexpr uint32_t OFF_Q = 4 * TILE;             // NSLOT slots
  static constexpr uint32_t OFF_DO = OFF_Q + NSLOT * TILE;
  static constexpr uint32_t OFF_DS = OFF_DO + NSLOT * TILE;
  static constexpr uint32_t OFF_STAT = OFF_DS + 2 * DS_REGION;  // per slot: lse*log2(e)[128], D[128]
  static constexpr uint32_t STAT_BYTES = 2u * 128u * 4u;
  // bf16 dQ tile on its way out (TMA store); dK and dV leave through the dS regions
  static constexpr uint32_t OFF_STAGE = OFF_STAT + NSLOT * STAT_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_STAGE + TILE;
  static constexpr uint32_t PAYLOAD = OFF_BAR + 512;
  static constexpr uint32_t SMEM = PAYLOAD + 1024;        // + alignment slack
  static_assert(SMEM <= 232448, "shared memory per block");
  static_assert(OFF_DS % 1024 == 0 && OFF_STAGE % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
  static constexpr int THREADS = 512;
  static constexpr int REG_COMPUTE = 152, REG_DQ = 88, REG_OTHER = 96;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TM_DQ = 256 + 2 * D;
  static_assert(TM_DQ + MAX_QT * D <= 512, "TMEM columns");
};

struct BwdHeadShared {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t qdo_full[3], slot_empty[3], stat_full[3];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dkv_full, acc_free, dq_full, dq_free, drain;
  uint64_t out_staged[3], out_free[3];  // [0], [1]: dV / dK through dS region 0 / 1; [2]: dQ stage
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdHeadShared) <= 512, "barrier block must fit its slot");

__device__ __forceinline__ float ex2h(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void drain_wait_h(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

// Writes one 128-row tile's row r (D bf16 given as D/2 packed words) into a
// shared-memory tile laid out as its TMA map expects: 128-byte rows with the
// 128-byte swizzle for D = 64, 64-byte rows with the 64-byte swizzle for D = 32.
template <int D>
__device__ __forceinline__ void stage_row(uint8_t* tile, int r, const uint32_t* w) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int pc = (D == 64) ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
    *reinterpret_cast<uint4*>(tile + r * (D * 2) + (pc << 4)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
}

// P^T for 32 query columns of one key row: p = 2^(s*c - lse2) with the
// negated statistic -lse2 read from shared memory, in fp32 pairs. MASKED:
// columns outside [lo, hi) (relative to this block) get weight exactly 0.
template <bool MASKED>
__device__ __forceinline__ void p_block(const uint32_t (&s)[32], const float* neg_lse2, uint64_t c2, int lo,
                                        int hi, uint64_t* P2) {
#pragma unroll
  for (int i4 = 0; i4 < 8; ++i4) {
    const float4 L = *reinterpret_cast<const float4*>(neg_lse2 + i4 * 4);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int col = i4 * 4 + u * 2;
      const uint64_t x2 = fma2(f2_pack(__uint_as_float(s[col]), __uint_as_float(s[col + 1])), c2,
                               u ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y));
      float x0, x1;
      f2_unpack(x2, x0, x1);
      if (MASKED) {
        if (col < lo || col >= hi) x0 = -INFINITY;
        if (col + 1 < lo || col + 1 >= hi) x1 = -INFINITY;
      }
      P2[i4 * 2 + u] = f2_pack(ex2h(x0), ex2h(x1));
    }
  }
}

// The key tiles [x, y] that read query tile t of a head with mb real keys
// (x = y = -1: none; then the tile's Q/dO slot is released and its dQ written
// as zero at the head's end). The rows that see any key are a prefix of the
// head (i < mb + wl with a left window, all rows otherwise, none when mb = 0),
// and the keys seen by consecutive such rows overlap, so the tile's rows see
// the one run of keys [lo(q0), hi(q_last)) with q_last its last such row; the
// key tiles meeting that run are exactly the key tiles whose query-tile range
// (query_range over the key tile) contains t.
__device__ __forceinline__ int2 key_tile_span(int t, int mb, int n, int causal, int wl, int wr) {
  const int q0 = t * 128;
  int q1 = min(q0 + 127, n - 1);
  if (wl >= 0) q1 = min(q1, mb + wl - 1);
  if (mb <= 0 || q1 < q0) return make_int2(-1, -1);
  int lo, hi, lo1, hi1;
  key_range(q0, mb, causal, wl, wr, lo, hi);
  key_range(q1, mb, causal, wl, wr, lo1, hi1);
  if (hi1 <= lo) return make_int2(-1, -1);
  return make_int2(lo / 128, (hi1 - 1) / 128);
}

// WIN: a restricted-attention window is set (otherwise both sides are open at
// compile time and the tile ranges reduce to the causal / padding ones).
template <int D, bool WIN>
__global__ void __launch_bounds__(512, 1)
attn_bwd_head_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const BwdHeadParams p) {
  using C = BwdHead<D>;
  extern __shared__ uint8_t smem_raw[];
  const Watchdog wd = p.wd;
  const int wl = WIN ? p.wl : -1, wr = WIN ? p.wr : -1;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad + C::PAYLOAD > C::SMEM) {
    if (threadIdx.x == 0) atomicCAS(wd.status, 0u, kDevLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  BwdHeadShared& sh = *reinterpret_cast<BwdHeadShared*>(smem + C::OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const int NQT = (p.n + 127) / 128;  // 1 or 2
  const int NKT = (p.m + 127) / 128;
  // query tiles [t0, t1) hold a row that sees some key of key tile kb (causal:
  // none wholly above the diagonal; key padding: none past the head's mb real
  // keys; a window: only those near the tile); t0 = t1 = NQT when none does
  auto q_tiles = [&](int kb, int mb, int& t0, int& t1) {
    const int k0 = kb * 128;
    t0 = t1 = NQT;
    if (k0 >= mb) return;
    int qlo, qhi;
    query_range(k0, min(k0 + 127, mb - 1), p.n, p.causal, wl, wr, qlo, qhi);
    if (qhi <= qlo) return;
    t0 = qlo / 128;
    t1 = (qhi + 127) / 128;
  };
  auto kb_span = [&](int t, int mb, int& f, int& l) {
    const int2 r = key_tile_span(t, mb, p.n, p.causal, wl, wr);
    f = r.x;
    l = r.y;
  };

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      mbar_init(&sh.kv_empty[s], 1);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&sh.qdo_full[s], 1);
      mbar_init(&sh.slot_empty[s], 1);
      mbar_init(&sh.stat_full[s], 64);
    }
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.p_full, 256);
    mbar_init(&sh.ds_full, 256);
    mbar_init(&sh.ds_empty, 1);
    mbar_init(&sh.dkv_full, 1);
    mbar_init(&sh.acc_free, 256);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 128);
    mbar_init(&sh.drain, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sh.out_staged[i], 128);
      mbar_init(&sh.out_free[i], 1);
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc<512>(&sh.tmem_base);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
    prefetch_tensormap(&tm_dq);
    prefetch_tensormap(&tm_dk);
    prefetch_tensormap(&tm_dv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);  // [slot][lse2 | D][128]

  if (warp >= 12) {
    reg_dealloc<C::REG_OTHER>();
  }
  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // per slot / set: bit = filled at least once, parity of the last fill
      uint32_t q_filled = 0, q_ph = 0, kv_filled = 0, kv_ph = 0;
      int k = 0, ki = 0;  // query tiles and key tiles loaded so far
      bool ok = true;
      for (int bh = blockIdx.x; ok && bh < p.BH; bh += gridDim.x) {
        // interleave so that the head's first query tile and first key tile come first
        const int steps = max(NQT, NKT);
        for (int step = 0; ok && step < steps; ++step) {
          if (step < NQT) {
            const int kk = k + step, slot = kk % C::NSLOT, use = kk / C::NSLOT;
            if (use >= 1 && !(ok = guarded_wait(&sh.slot_empty[slot], (use - 1) & 1, abort_flag, wd, kSiteBwdFree)))
              break;
            mbar_arrive_expect_tx(&sh.qdo_full[slot], 2 * C::TILE);
            tma_load_3d(smem + C::OFF_Q + slot * C::TILE, &tm_q, &sh.qdo_full[slot], 0, step * 128, bh);
            tma_load_3d(smem + C::OFF_DO + slot * C::TILE, &tm_do, &sh.qdo_full[slot], 0, step * 128, bh);
            q_filled |= 1u << slot;
            q_ph = (q_ph & ~(1u << slot)) | (static_cast<uint32_t>(use & 1) << slot);
          }
          if (step < NKT) {
            const int set = ki & 1, use = ki >> 1;
            if (use >= 1 && !(ok = guarded_wait(&sh.kv_empty[set], (use - 1) & 1, abort_flag, wd, kSiteBwdFree)))
              break;
            mbar_arrive_expect_tx(&sh.kv_full[set], 2 * C::TILE);
            tma_load_3d(smem + C::OFF_K + set * C::TILE, &tm_k, &sh.kv_full[set], 0, step * 128, bh);
            tma_load_3d(smem + C::OFF_V + set * C::TILE, &tm_v, &sh.kv_full[set], 0, step * 128, bh);
            kv_filled |= 1u << set;
            kv_ph = (kv_ph & ~(1u << set)) | (static_cast<uint32_t>(use & 1) << set);
            ++ki;
          }
        }
        k += NQT;
      }
      // Let every copy this thread started land before shared memory is released.
      for (int s = 0; s < C::NSLOT; ++s)
        if ((q_filled >> s) & 1u) drain_wait_h(&sh.qdo_full[s], (q_ph >> s) & 1u, wd);
      for (int s = 0; s < 2; ++s)
        if ((kv_filled >> s) & 1u) drain_wait_h(&sh.kv_full[s], (kv_ph >> s) & 1u, wd);
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    const uint32_t id_s = idesc_bf16_f32(128, 128, false, false) | (p.neg ? (1u << 13) : 0u);
    const uint32_t id_dp = idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_kv = idesc_bf16_f32(128, D, false, true);   // dV, dK: B = dO / Q, MN-major
    const uint32_t id_dq = idesc_bf16_f32(128, D, true, true);    // dQ: A = dS (MN-major), B = K (MN-major)
    // X = A_tile (rows in TMEM lanes) times B_tile^T, both K-major over d.
    auto issue_kmajor = [&](uint32_t d_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint64_t da = smem_desc(a_base + k * 32, 16, C::SBO, C::SWZ);
        const uint64_t db = smem_desc(b_base + k * 32, 16, C::SBO, C::SWZ);
        mma_ss(d_tmem, da, db, idesc, k > 0 ? 1u : 0u);
      }
    };
    // B operand: a [128 rows][D] tile read MN-major, K = 16 rows per step.
    auto b_mn = [&](uint32_t base, int k) { return smem_desc(base + k * 16 * C::ATOM * 2, C::TILE, C::SBO, C::SWZ); };
    auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, guarded_wait(bar, parity, abort_flag, wd, site));
    };
    bool ok = true;
    int g = 0, k = 0, ki = 0, li = 0;
    for (int bh = blockIdx.x; ok && bh < p.BH; bh += gridDim.x, ++li) {
      const int mb = head_keys(p.kv_len, bh, p.h, p.m);  // real keys of this head
      // dq_free is waited once per head, in order: before the head's first dQ
      // product, or at the head's end when it has none
      bool dq_waited = (li == 0);
      int f0, l0, f1 = -1, l1 = -1;  // key tiles reading query tiles 0 and 1
      kb_span(0, mb, f0, l0);
      if (NQT > 1) kb_span(1, mb, f1, l1);
      for (int kb = 0; ok && kb < NKT; ++kb, ++ki) {
        const int set = ki & 1;
        const uint32_t sK = smem_u32(smem + C::OFF_K + set * C::TILE);
        const uint32_t sV = smem_u32(smem + C::OFF_V + set * C::TILE);
        if (!(ok = wait_all(&sh.kv_full[set], (ki >> 1) & 1, kSiteBwdLoad))) break;
        int t0, t1;
        q_tiles(kb, mb, t0, t1);
        const int T = t1 - t0;
        // acc_free is waited once per key tile, in order: below before the
        // first dV product, or here for a key tile without query tiles
        if (T == 0 && ki >= 1 && !(ok = wait_all(&sh.acc_free, (ki - 1) & 1, kSiteBwdFinal))) break;
        if (T > 0) {
          const int kk0 = k + t0;
          if (!(ok = wait_all(&sh.qdo_full[kk0 % C::NSLOT], (kk0 / C::NSLOT) & 1, kSiteBwdLoad))) break;
          if (lane == 0) {
            tc_fence_after();
            issue_kmajor(tmem + C::TM_S, sK, sQ + (kk0 % C::NSLOT) * C::TILE, id_s);
            mma_commit(&sh.s_full);
            issue_kmajor(tmem + C::TM_DP, sV, sDO + (kk0 % C::NSLOT) * C::TILE, id_dp);
            mma_commit(&sh.dp_full);
          }
          __syncwarp();
        }
        for (int t = t0; ok && t < t1; ++t) {
          const int gt = g + (t - t0);
          const int kk = k + t, slot = kk % C::NSLOT;
          const uint32_t q_off = slot * C::TILE;
          // dV += P^T dO; P^T (bf16) sits in TMEM columns [0,32) and [64,96) of S^T,
          // one block per compute warpgroup (queries 0..63 and 64..127)
          if (!(ok = wait_all(&sh.p_full, gt & 1, kSiteBwdS))) break;
          // The first dV product of a key tile overwrites the accumulators: the
          // previous key tile's epilogue must have read dK and dV out of TMEM.
          // (Waiting here, not at the key tile's start, lets S^T and dP^T of
          // this key tile overlap that epilogue.)
          if (t == t0 && ki >= 1 && !(ok = wait_all(&sh.acc_free, (ki - 1) & 1, kSiteBwdFinal))) break;
          if (lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              mma_ts(tmem + C::TM_DV, tmem + C::TM_S + (q >> 2) * 64 + (q & 3) * 8, b_mn(sDO + q_off, q), id_kv,
                     (t > t0 || q > 0) ? 1u : 0u);
          }
          __syncwarp();
          // next S^T while the compute warps form dS
          if (t + 1 < t1) {
            const int kn = kk + 1;
            if (!(ok = wait_all(&sh.qdo_full[kn % C::NSLOT], (kn / C::NSLOT) & 1, kSiteBwdLoad))) break;
            if (lane == 0) {
              issue_kmajor(tmem + C::TM_S, sK, sQ + (kn % C::NSLOT) * C::TILE, id_s);
              mma_commit(&sh.s_full);
            }
            __syncwarp();
          }
          if (!(ok = wait_all(&sh.ds_full, gt & 1, kSiteBwdDS))) break;
          // the head's first dQ product overwrites the previous head's dQ
          if (!dq_waited) {
            if (!(ok = wait_all(&sh.dq_free, (li - 1) & 1, kSiteBwdDQ))) break;
            dq_waited = true;
          }
          const bool dq_acc = kb > (t ? f1 : f0);  // query tile t's first dQ product starts it
          if (lane == 0) {
            tc_fence_after();
            // dK += dS^T Q : A = dS^T (K-major over queries), B = Q (MN-major)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint64_t da = smem_desc(sDS + (q >> 2) * C::DS_REGION + (q & 3) * 32, 16, 1024, 2);
              mma_ss(tmem + C::TM_DK, da, b_mn(sQ + q_off, q), id_kv, (t > t0 || q > 0) ? 1u : 0u);
            }
            // dQ_t += dS K : A = dS (MN-major: queries contiguous), B = K (MN-major)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint64_t da = smem_desc(sDS + q * 16 * 128, C::DS_REGION, 1024, 2);
              mma_ss(tmem + C::TM_DQ + t * D, da, b_mn(sK, q), id_dq, (dq_acc || q > 0) ? 1u : 0u);
            }
            mma_commit(&sh.ds_empty);
            if (kb == (t ? l1 : l0)) mma_commit(&sh.slot_empty[slot]);  // no later product reads this slot
          }
          __syncwarp();
          if (t + 1 < t1) {
            const int kn = kk + 1;
            if (lane == 0) {
              issue_kmajor(tmem + C::TM_DP, sV, sDO + (kn % C::NSLOT) * C::TILE, id_dp);
              mma_commit(&sh.dp_full);
            }
            __syncwarp();
          }
        }
        if (!ok) break;
        if (lane == 0) {
          mma_commit(&sh.dkv_full);
          mma_commit(&sh.kv_empty[set]);
        }
        __syncwarp();
        g += T;
      }
      if (!ok) break;
      if (!dq_waited && !(ok = wait_all(&sh.dq_free, (li - 1) & 1, kSiteBwdDQ))) break;
      if (lane == 0) {
        // query tiles that no key tile read (a head without real keys) free their slots here
        for (int t = 0; t < NQT; ++t)
          if ((t ? l1 : l0) < 0) mma_commit(&sh.slot_empty[(k + t) % C::NSLOT]);
        mma_commit(&sh.dq_full);  // every dQ product of this head
      }
      __syncwarp();
      k += NQT;
    }
    if (lane == 0) mma_commit(&sh.drain);
    __syncwarp();
    drain_wait_h(&sh.drain, 0, wd);
  } else if (warp >= 14) {
    // ------------------------------------------------------------ per-row statistics
    // Thread u handles query rows u and u + 64 of every query tile: D_i = dO_i . O_i
    // in fp32 from the bf16 rows, and lse_i * log2(e); rows past n get D = 0
    // and lse = +inf, so that their weights vanish.
    const int u = tid - 448;
    int k = 0;
    bool ok = true;
    for (int bh = blockIdx.x; ok && bh < p.BH; bh += gridDim.x) {
      for (int t = 0; t < NQT; ++t) {
        const int kk = k + t, slot = kk % C::NSLOT;
        // The statistics depend only on O, dO and lse in global memory: they are
        // formed before the wait for the slot, so that their loads (O comes from
        // HBM) overlap it instead of following it at every head's start.
        float nlse2[2], dsum[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int row = t * 128 + u + 64 * half;
          float ds = 0.f, lse2 = INFINITY;
          if (row < p.n) {
            const size_t off = (static_cast<size_t>(bh) * p.n + row) * D;
            const uint4* o4 = reinterpret_cast<const uint4*>(p.o + off);
            const uint4* d4 = reinterpret_cast<const uint4*>(p.dO + off);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
              const uint4 a = o4[c], b = d4[c];
              const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const float2 x = unpack_bf16x2(av[w]), y = unpack_bf16x2(bv[w]);
                ds = fmaf(x.x, y.x, ds);
                ds = fmaf(x.y, y.y, ds);
              }
            }
            // a row that saw no key (lse = -inf, O = 0) keeps lse2 = +inf: weight 0
            const float lse = p.lse[static_cast<size_t>(bh) * p.n + row];
            if (lse > -INFINITY) lse2 = lse * kLog2eH;
          }
          nlse2[half] = -lse2;
          dsum[half] = ds;
        }
        // the slot's previous statistics are no longer read once its new tile has landed
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.qdo_full[slot], (kk / C::NSLOT) & 1, abort_flag, wd,
                                                  kSiteBwdLoad));
        if (!ok) break;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          stat[slot * 256 + u + 64 * half] = nlse2[half];
          stat[slot * 256 + 128 + u + 64 * half] = dsum[half];
        }
        mbar_arrive(&sh.stat_full[slot]);
      }
      k += NQT;
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P, dS, dK/dV epilogue
    reg_alloc<C::REG_COMPUTE>();
    const int h = warp >> 2;
    const int col0 = 64 * h;
    const int r = tid & 127;                            // key row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::TM_S + col0;
    const uint32_t t_dp = tmem + lane_base + C::TM_DP + col0;
    const float c = p.c;
    uint8_t* ds_row = smem + C::OFF_DS + h * C::DS_REGION + r * 128;
    const int sw = r & 7;
    bool ok = true;
    int g = 0, k = 0, ki = 0;
    // Region h carried the previous key tile's dV / dK out. Thread 0 issued that
    // TMA store and checks that it has read the region only when this key tile
    // first writes there (its first dS, or its own output when no query tile
    // reads it), so that the group forms the key tile's first P meanwhile.
    bool store_pending = false;
    auto region_free = [&]() -> bool {
      if (ki == 0) return true;
      if (r == 0 && store_pending) {
        bulk_wait_read_all();
        mbar_arrive(&sh.out_free[h]);
        store_pending = false;
      }
      return __all_sync(0xffffffffu, guarded_wait(&sh.out_free[h], (ki - 1) & 1, abort_flag, wd, kSiteBwdFinal));
    };
    for (int bh = blockIdx.x; ok && bh < p.BH; bh += gridDim.x) {
      const int mb = head_keys(p.kv_len, bh, p.h, p.m);  // real keys of this head
      for (int kb = 0; ok && kb < NKT; ++kb, ++ki) {
        const int key = kb * 128 + r;
        int t0, t1;
        q_tiles(kb, mb, t0, t1);
        const int T = t1 - t0;
        int qlo, qhi;  // query rows that see this key
        query_range(key, key, p.n, p.causal, wl, wr, qlo, qhi);
        for (int t = t0; t < t1; ++t) {
          const int gt = g + (t - t0);
          const int kk = k + t, slot = kk % C::NSLOT;
          const int q_row0 = t * 128;
          // queries [lo, hi) of this tile may attend to this key
          const int lo = max(0, qlo - q_row0);
          const int hi = (key < mb) ? min(128, qhi - q_row0) : 0;
          const bool masked = __any_sync(0xffffffffu, lo > col0 || hi < col0 + 64);
          ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full, gt & 1, abort_flag, wd, kSiteBwdS) &&
                                           guarded_wait(&sh.stat_full[slot], (kk / C::NSLOT) & 1, abort_flag, wd,
                                                        kSiteBwdLoad));
          if (!ok) break;
          tc_fence_after();
          const float* nlse2_s = stat + slot * 256 + col0;  // -lse*log2(e) per query column
          const float* D_s = stat + slot * 256 + 128 + col0;
          // P^T in fp32 pairs for dS below; rounded to bf16 for the dV product
          uint64_t P2[32];
          {
            uint32_t s[2][32];
            tmem_ld32(t_s, s[0]);
            tmem_ld32(t_s + 32, s[1]);
            tmem_ld_wait();
            const uint64_t c2 = f2_pack(c, c);
            if (masked) {
              p_block<true>(s[0], nlse2_s, c2, lo - col0, hi - col0, P2);
              p_block<true>(s[1], nlse2_s + 32, c2, lo - col0 - 32, hi - col0 - 32, P2 + 16);
            } else {
              p_block<false>(s[0], nlse2_s, c2, 0, 32, P2);
              p_block<false>(s[1], nlse2_s + 32, c2, 0, 32, P2 + 16);
            }
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2_pair(P2[q * 16 + i]);
            tmem_st16(t_s + q * 16, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sh.p_full);
          // dS = P (dP - D)
          ok = __all_sync(0xffffffffu, guarded_wait(&sh.dp_full, gt & 1, abort_flag, wd, kSiteBwdDP));
          if (!ok) break;
          tc_fence_after();
          if (gt >= 1) {
            ok = __all_sync(0xffffffffu, guarded_wait(&sh.ds_empty, (gt - 1) & 1, abort_flag, wd, kSiteBwdDS));
            if (!ok) break;
          }
          if (t == t0 && !(ok = region_free())) break;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t dp[32];
            tmem_ld32(t_dp + q * 32, dp);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 Dv = *reinterpret_cast<const float4*>(D_s + q * 32 + i4 * 4);
              const uint64_t a = mul2(P2[q * 16 + i4 * 2],
                                      sub2(f2_pack(__uint_as_float(dp[i4 * 4]), __uint_as_float(dp[i4 * 4 + 1])),
                                           f2_pack(Dv.x, Dv.y)));
              const uint64_t b = mul2(P2[q * 16 + i4 * 2 + 1],
                                      sub2(f2_pack(__uint_as_float(dp[i4 * 4 + 2]), __uint_as_float(dp[i4 * 4 + 3])),
                                           f2_pack(Dv.z, Dv.w)));
              pk[i4 * 2 + 0] = pack_bf16x2_pair(a);
              pk[i4 * 2 + 1] = pack_bf16x2_pair(b);
            }
            // these 32 queries are 16-byte chunks 4q..4q+3 of this row of region h
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const int chunk = q * 4 + ch;
              *reinterpret_cast<uint4*>(ds_row + ((chunk ^ sw) << 4)) =
                  make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&sh.ds_full);
        }
        if (!ok) break;
        // epilogue: group 0 writes dV, group 1 writes scale * dK, rows of this key tile.
        // Taken for key tiles without query tiles too, so that these warps stay
        // at most one key tile ahead of the MMA warp.
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.dkv_full, ki & 1, abort_flag, wd, kSiteBwdFinal));
        if (!ok) break;
        tc_fence_after();
        uint32_t w[D / 2];
        const float mul = h ? p.scale : 1.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          if (T > 0) {
            tmem_ld32(tmem + lane_base + (h ? C::TM_DK : C::TM_DV) + q * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[q * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        }
        // the accumulators are read: the next key tile's dV / dK may start
        tc_fence_before();
        mbar_arrive(&sh.acc_free);
        // a key tile that no query tile reads wrote no dS: the region is first
        // written here
        if (T == 0 && !(ok = region_free())) break;
        // stage this row in region h and let one thread store the tile (rows
        // past m are clipped by the tensor map)
        uint8_t* region = smem + C::OFF_DS + h * C::DS_REGION;
        stage_row<D>(region, r, w);
        fence_proxy_async_smem();
        mbar_arrive(&sh.out_staged[h]);
        if (r == 0) {
          if (guarded_wait(&sh.out_staged[h], ki & 1, abort_flag, wd, kSiteBwdFinal)) {
            tma_store_3d(h ? &tm_dk : &tm_dv, region, 0, kb * 128, bh);
            tma_store_commit();
          }
          store_pending = true;  // released where the next key tile first writes the region
        }
        g += T;
      }
      k += NQT;
    }
  } else {
    // ------------------------------------------------------------ dQ epilogue (warps 8-11)
    reg_dealloc<C::REG_DQ>();
    const int r = tid - 256;                           // query row within a tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int li = 0, ns = 0;  // heads done, dQ tiles stored
    for (int bh = blockIdx.x; bh < p.BH; bh += gridDim.x, ++li) {
      const bool ok = __all_sync(0xffffffffu, guarded_wait(&sh.dq_full, li & 1, abort_flag, wd, kSiteBwdDQ));
      if (!ok) break;
      tc_fence_after();
      uint8_t* stage = smem + C::OFF_STAGE;
      const int mb = head_keys(p.kv_len, bh, p.h, p.m);
      bool live = true;
      for (int t = 0; live && t < NQT; ++t, ++ns) {
        // a query tile that no key tile reads (a head without real keys, rows
        // whose windows miss every key) has no dQ product: its dQ is zero
        // (TMEM still holds an earlier head's)
        int f, l;
        kb_span(t, mb, f, l);
        const bool empty = f < 0;
        uint32_t w[D / 2];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          if (!empty) {
            tmem_ld32(tmem + lane_base + C::TM_DQ + t * D + q * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[q * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]) * p.scale, __uint_as_float(v[2 * i + 1]) * p.scale);
        }
        if (t == NQT - 1) {
          // every dQ accumulator of this head is read: the next head may overwrite them
          tc_fence_before();
          mbar_arrive(&sh.dq_free);
        }
        // the previous tile's store must have read the stage
        if (ns >= 1) {
          live = __all_sync(0xffffffffu, guarded_wait(&sh.out_free[2], (ns - 1) & 1, abort_flag, wd, kSiteBwdDQ));
          if (!live) break;
        }
        stage_row<D>(stage, r, w);
        fence_proxy_async_smem();
        mbar_arrive(&sh.out_staged[2]);
        if (r == 0) {
          if (guarded_wait(&sh.out_staged[2], ns & 1, abort_flag, wd, kSiteBwdDQ)) {
            tma_store_3d(&tm_dq, stage, 0, t * 128, bh);  // rows past n are clipped
            tma_store_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&sh.out_free[2]);
        }
      }
      if (!live) break;
    }
  }

  // bulk stores issued by this thread must complete before the CTA exits
  if ((warp == 0 || warp == 4 || warp == 8) && lane == 0) tma_store_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int D, bool WIN>
cudaError_t launch_bwd_head_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                              const CUtensorMap& tdv, const BwdHeadParams& p, cudaStream_t stream) {
  using C = BwdHead<D>;
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_bwd_head_kernel<D, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  static int regs_per_thread[64] = {0};
  static int sm_count[64] = {0};
  if (regs_per_thread[dev & 63] == 0) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, attn_bwd_head_kernel<D, WIN>)) != cudaSuccess) return e;
    regs_per_thread[dev & 63] = fa.numRegs;
  }
  // setmaxnreg.inc waits until registers are free: the split must fit in the
  // registers the CTA is launched with, or the kernel would never proceed.
  if (regs_per_thread[dev & 63] * C::THREADS < 128 * (2 * C::REG_COMPUTE + C::REG_DQ + C::REG_OTHER))
    return cudaErrorInvalidConfiguration;
  if (sm_count[dev & 63] == 0) {
    int c = 0;
    if ((e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    sm_count[dev & 63] = c > 0 ? c : 1;
  }
  const int grid = p.BH < sm_count[dev & 63] ? p.BH : sm_count[dev & 63];
  prof_begin(kKindBwdMain, stream);
  attn_bwd_head_kernel<D, WIN><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
  e = cudaGetLastError();
  prof_end(kKindBwdMain, stream);
  return e;
}

}  // namespace

bool bwd_head_supported(int n, int d) { return n >= 1 && n <= 256 && (d == 32 || d == 64); }

cudaError_t launch_bwd_head(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdHeadParams& p, cudaStream_t stream) {
  const bool win = p.wl >= 0 || p.wr >= 0;
  switch (d) {
    case 32:
      return win ? launch_bwd_head_d<32, true>(tq, tk, tv, tdo, tdq, tdk, tdv, p, stream)
                 : launch_bwd_head_d<32, false>(tq, tk, tv, tdo, tdq, tdk, tdv, p, stream);
    case 64:
      return win ? launch_bwd_head_d<64, true>(tq, tk, tv, tdo, tdq, tdk, tdv, p, stream)
                 : launch_bwd_head_d<64, false>(tq, tk, tv, tdo, tdq, tdk, tdv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
