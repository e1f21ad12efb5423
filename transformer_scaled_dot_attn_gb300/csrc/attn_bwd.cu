// Backward kernels: dQ, dK, dV of L = sum(dO * O) for O = softmax(Q K^T * scale) V.
//
// The pages train the model (§5 of "Attention Is All You Need") but never
// write the derivative of eq. (1) out; it is the analytic one:
//   P_ij = exp(scale q_i.k_j - lse_i)         (recomputed, never stored)
//   D_i  = sum_c dO_ic O_ic
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
// Masked pairs (key j after query i, §3.2.3) have P_ij = 0 and drop out.
//
// Three launches on the caller's stream:
//   pre   D_i, lse_i * log2(e) into padded rows of the workspace; zero the fp32
//         dQ accumulator. Bandwidth bound.
//   main  one CTA per (head, 128-key tile j). K_j and V_j stay in shared
//         memory; 128-query tiles i stream through a two-stage TMA ring.
//         Five tcgen05 products per tile, all with 128 TMEM lanes:
//           S^T  = K_j Q_i^T        (lanes: keys)            -> TMEM
//           dP^T = V_j dO_i^T                                 -> TMEM
//           dV_j += P^T dO_i        (P^T bf16 in TMEM, aliasing S^T)
//           dK_j += dS^T Q_i        (dS^T bf16 in shared memory, K-major view)
//           dQ_i  = dS K_j          (same buffer read as an MN-major operand)
//         warps 0-7  two warpgroups, one thread per key row each, on
//                    disjoint query columns: P, dS, and the dK/dV epilogue.
//         warps 8-11 one thread per query row: add dQ_i into the fp32
//                    accumulator with TMA reduce-adds.
//         warp 12    TMA producer (tiles, and the per-row statistics by
//                    bulk copy); warps 13 and 14 the two MMA issuers, one
//                    for S^T and dV, one for dP^T, dQ and dK.
//   post  dQ = bf16(scale * accumulator).
//
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D),
// dQ [256+2D,256+3D) for D <= 64; for D = 128 dQ reuses the dP^T columns.
// dQ leaves the SM by TMA reduce-adds of a staged fp32 tile (d = 128 stages
// it through the dS buffer, two rounds of 64 columns).
// Warps (512 threads): 0-3 and 4-7 the two compute warpgroups (query columns
// 0..63 / 64..127 of every tile), 8-11 dQ accumulation, 12 TMA producer,
// 13 and 14 MMA issuers; registers split 152 / 152 / 96 / 88 with setmaxnreg.
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr float kLog2e = 1.4426950408889634074f;

// ---------------------------------------------------------------- pre

// One group of D/8 lanes per row: each lane reads 8 bf16 of O and dO.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const BwdPreParams p) {
  constexpr int LPR = D / 8;           // lanes per row
  constexpr int RPB = 256 / LPR;       // rows per block
  const long long row = static_cast<long long>(blockIdx.x) * RPB + threadIdx.x / LPR;
  const int sub = threadIdx.x % LPR;
  const long long total = static_cast<long long>(p.BH) * p.n_pad;
  float dot = 0.f;
  bool valid = false;
  long long bh = 0, i = 0;
  if (row < total) {
    bh = row / p.n_pad;
    i = row - bh * p.n_pad;
    valid = i < p.n;
    if (valid) {
      const size_t off = (static_cast<size_t>(bh) * p.n + i) * D + sub * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(p.o + off);
      const uint4 b = *reinterpret_cast<const uint4*>(p.dO + off);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(a2[t]);
        const float2 y = __bfloat1622float2(b2[t]);
        dot = fmaf(x.x, y.x, dot);
        dot = fmaf(x.y, y.y, dot);
      }
    }
    // zero this row's slice of the dQ accumulator (D floats = D/4 float4, 2 per lane)
    float4* acc = reinterpret_cast<float4*>(p.dq_acc + static_cast<size_t>(row) * D) + sub * 2;
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off, LPR);
  if (row < total && sub == 0) {
    p.Dsum[row] = valid ? dot : 0.f;
    // -lse * log2(e), the exponent offset of P; rows past n and rows that saw no
    // key (lse = -inf) get -inf: weight 0
    const float lse = valid ? p.lse[static_cast<size_t>(bh) * p.n + i] : -INFINITY;
    p.lse2[row] = (lse > -INFINITY) ? -lse * kLog2e : -INFINITY;
  }
}

// ---------------------------------------------------------------- post

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const BwdPostParams p) {
  constexpr int CPR = D / 8;  // 8-element chunks per row
  const long long idx = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  const long long total = static_cast<long long>(p.BH) * p.n * CPR;
  if (idx >= total) return;
  const long long row = idx / CPR;
  const int ch = static_cast<int>(idx - row * CPR);
  const long long bh = row / p.n;
  const long long i = row - bh * p.n;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc + (static_cast<size_t>(bh) * p.n_pad + i) * D) + ch * 2;
  const float4 a = src[0], b = src[1];
  uint4 out;
  out.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
  out.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
  out.z = pack_bf16x2(b.x * p.scale, b.y * p.scale);
  out.w = pack_bf16x2(b.z * p.scale, b.w * p.scale);
  reinterpret_cast<uint4*>(p.dq + static_cast<size_t>(row) * D)[ch] = out;
}

// ---------------------------------------------------------------- main

template <int D>
struct Bwd {
  static constexpr int ATOM = (D >= 64) ? 64 : D;
  static constexpr int NATOM = D / ATOM;
  static constexpr uint32_t SWZ = (D >= 64) ? 2u : 4u;
  static constexpr uint32_t SBO = 8u * ATOM * 2u;
  static constexpr uint32_t TILE = 128u * D * 2u;
  static constexpr uint32_t BOX = 128u * ATOM * 2u;
  static constexpr uint32_t DS_REGION = 128u * 64u * 2u;
  // K/V tiles: two sets for d <= 64 so the next work item's keys load while
  // the current one finishes; one set for d = 128 (shared memory is full).
  // Q / dO ring: three stages for d <= 64 (a query tile's loads take about half
  // a tile's time to land), two for d = 128 (shared memory is full). K/V: two
  // sets for d = 32 so the next item's keys load early; one otherwise (d = 64
  // gives its second set to the third Q / dO stage).
  static constexpr int QS = (D <= 64) ? 3 : 2;
  static constexpr int KV_SETS = (D <= 32) ? 2 : 1;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = KV_SETS * TILE;
  static constexpr uint32_t OFF_Q = 2 * KV_SETS * TILE;          // QS stages
  static constexpr uint32_t OFF_DO = OFF_Q + QS * TILE;          // QS stages
  static constexpr uint32_t OFF_DS = OFF_DO + QS * TILE;         // dS^T: 2 regions [128 keys][64 queries]
  static constexpr uint32_t OFF_STAT = OFF_DS + 2 * DS_REGION;   // per stage: lse*log2(e)[128], D[128]
  static constexpr uint32_t STAT_BYTES = 2u * 128u * 4u;
  // The fp32 dQ tile is staged in shared memory (128-byte swizzled boxes of
  // 32 columns) and added into the accumulator by TMA reduces. d <= 64 has a
  // staging area of its own; d = 128 has no room left and stages through the
  // dS buffer (free once dK and dQ have read it) in two rounds of 64 columns,
  // releasing the buffer to the next tile's dS when the reduces have read it.
  static constexpr uint32_t DQ_BOX = 128u * 32u * 4u;
  static constexpr bool DQ_IN_DS = (D > 64);
  static constexpr int DQ_ROUNDS = DQ_IN_DS ? 2 : 1;
  static constexpr int DQ_BOXES_PER_ROUND = (D / 32) / DQ_ROUNDS;
  static constexpr uint32_t OFF_DQS = OFF_STAT + QS * STAT_BYTES;
  static constexpr uint32_t DQS_BYTES = DQ_IN_DS ? 0u : (D / 32) * DQ_BOX;
  static constexpr uint32_t OFF_BAR = OFF_DQS + DQS_BYTES;
  static constexpr uint32_t PAYLOAD = OFF_BAR + 256;
  static constexpr uint32_t SMEM_LIMIT = 232448;                 // opt-in maximum per block
  // + up to 1 KB to align the tiles; for D = 128 only what fits under the limit
  static constexpr uint32_t SMEM = (PAYLOAD + 1024 <= SMEM_LIMIT) ? PAYLOAD + 1024 : SMEM_LIMIT;
  static constexpr int THREADS = 512;
  // d <= 64: the dV / dK tile (128 rows) fits a dS region and leaves by TMA store
  static constexpr bool STAGE_OUT = (D <= 64);
  static_assert(OFF_DS % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
  // setmaxnreg split (registers per thread): compute, dQ, producer/MMA warpgroups.
  static constexpr int REG_COMPUTE = 152, REG_DQ = 96, REG_OTHER = 88;
  static constexpr bool ALIAS_DQ = (D > 64);
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr uint32_t TM_DQ = ALIAS_DQ ? 128u : (256u + 2u * D);
};

struct BwdShared {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t qdo_full[3], qdo_empty[3];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full, dq_empty, dkv_full, acc_free, drain, drain_b;
  uint64_t dk_done;  // d = 128: the dK product has read dS (the dQ staging may overwrite it)
  uint64_t out_staged[2], out_free[2];  // d <= 64: dV / dK leave through dS region 0 / 1
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdShared) <= 256, "barrier block must fit its slot");

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void drain_wait_b(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

// WIN: a restricted-attention window is set (otherwise both sides are open at
// compile time and the tile ranges reduce to the causal / padding ones).
template <int D, bool WIN>
__global__ void __launch_bounds__(512, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using C = Bwd<D>;
  extern __shared__ uint8_t smem_raw[];
  const Watchdog wd = p.wd;
  const int wl = WIN ? p.wl : -1, wr = WIN ? p.wr : -1;
  // The tiles need 1024-byte alignment (128-byte swizzle atoms). The kernel
  // declares no static shared memory, so the dynamic window starts aligned in
  // practice; if it ever did not leave room, report it and do nothing.
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad + C::PAYLOAD > C::SMEM) {
    if (threadIdx.x == 0) atomicCAS(wd.status, 0u, kDevLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  BwdShared& sh = *reinterpret_cast<BwdShared*>(smem + C::OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const int n_qt = (p.n + 127) / 128;
  // Work item it = (key tile kb, head bh). Every CTA takes items it =
  // blockIdx.x, blockIdx.x + gridDim.x, ...; the query tiles of an item:
  // [i_start, i_start + T), those with a row that sees one of its keys
  // (causal: none wholly above the key tile; a window: only those near it).
  // Causal: key-tile major, so that the items with the most query tiles come
  // first; all CTAs of a head walk the query tiles in the same order (the
  // streamed Q and dO tiles come from DRAM once, then from L2). Otherwise head
  // major (p.head_major): the CTAs running at once cover a few heads, and each
  // item starts at its own query tile (rot = kb mod T) so that the CTAs of a
  // head add into different dQ tiles at a time; measured 3-4 % faster at d = 64
  // on GB300 (with the order read from the parameters: the same order fixed at
  // compile time measured no faster than key-tile major). Key padding: a key
  // tile wholly past the head's real keys has no query tiles (its dK, dV rows
  // are zero).
  auto item_of = [&](int it, int& bh, int& kb, int& i_start, int& T, int& rot) {
    if (p.head_major) {
      bh = it / p.num_kblocks;
      kb = it - bh * p.num_kblocks;
    } else {
      kb = it / p.BH;
      bh = it - kb * p.BH;
    }
    rot = 0;
    const int mb = head_keys(p.kv_len, bh, p.h, p.m);
    i_start = n_qt;
    T = 0;
    const int k0 = kb * 128;
    if (k0 >= mb) return;
    int qlo, qhi;
    query_range(k0, min(k0 + 127, mb - 1), p.n, p.causal, wl, wr, qlo, qhi);
    if (qhi <= qlo) return;
    i_start = qlo / 128;
    T = (qhi + 127) / 128 - i_start;
    if (p.head_major) rot = kb % T;
  };
  // the item's t-th query tile in its walk
  auto q_tile = [&](int i_start, int T, int rot, int t) {
    return i_start + (t + rot < T ? t + rot : t + rot - T);
  };

  if (tid == 0) {
    for (int s = 0; s < C::KV_SETS; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      mbar_init(&sh.kv_empty[s], 2);  // both MMA issuers read the set
    }
    for (int s = 0; s < C::QS; ++s) {
      mbar_init(&sh.qdo_full[s], 1);
      mbar_init(&sh.qdo_empty[s], 2);  // both MMA issuers read the stage
    }
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.p_full, 256);
    mbar_init(&sh.ds_full, 256);
    mbar_init(&sh.ds_empty, 1);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_empty, 128);
    mbar_init(&sh.dkv_full, 2);  // dV (issuer A) and dK (issuer B) complete
    mbar_init(&sh.acc_free, 256);
    mbar_init(&sh.drain, 1);
    mbar_init(&sh.drain_b, 1);
    mbar_init(&sh.dk_done, 1);
    for (int i = 0; i < 2; ++i) {
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
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);  // [stage][-lse2 | D][128]

  if (warp >= 12) {
    reg_dealloc<C::REG_OTHER>();
  }
  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // parity of the last fill of each K/V set and each Q/dO stage (-1: never filled);
      // scalars rather than arrays so that they stay in registers
      int kv_last0 = -1, kv_last1 = -1, q_last0 = -1, q_last1 = -1, q_last2 = -1;
      int g = 0, li = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < p.num_items; it += gridDim.x, ++li) {
        int bh, kb, i_start, T, rot;
        item_of(it, bh, kb, i_start, T, rot);
        const int set = li % C::KV_SETS, use = li / C::KV_SETS;
        if (li >= C::KV_SETS && !guarded_wait(&sh.kv_empty[set], (use - 1) & 1, abort_flag, wd, kSiteBwdFree)) break;
        mbar_arrive_expect_tx(&sh.kv_full[set], 2 * C::TILE);
        for (int a = 0; a < C::NATOM; ++a) {
          tma_load_3d(smem + C::OFF_K + set * C::TILE + a * C::BOX, &tm_k, &sh.kv_full[set], a * C::ATOM,
                      kb * 128, bh);
          tma_load_3d(smem + C::OFF_V + set * C::TILE + a * C::BOX, &tm_v, &sh.kv_full[set], a * C::ATOM,
                      kb * 128, bh);
        }
        if (set == 0) kv_last0 = use & 1; else kv_last1 = use & 1;
        const float* lse2_h = p.lse2 + static_cast<size_t>(bh) * p.n_pad;
        const float* D_h = p.Dsum + static_cast<size_t>(bh) * p.n_pad;
        for (int t = 0; t < T; ++t, ++g) {
          const int st = g % C::QS;
          const uint32_t ph = (g / C::QS) & 1;
          if (g >= C::QS && !guarded_wait(&sh.qdo_empty[st], ph ^ 1, abort_flag, wd, kSiteBwdFree)) {
            ok = false;
            break;
          }
          const int q_row = q_tile(i_start, T, rot, t) * 128;
          mbar_arrive_expect_tx(&sh.qdo_full[st], 2 * C::TILE + C::STAT_BYTES);
          for (int a = 0; a < C::NATOM; ++a) {
            tma_load_3d(smem + C::OFF_Q + st * C::TILE + a * C::BOX, &tm_q, &sh.qdo_full[st], a * C::ATOM, q_row, bh);
            tma_load_3d(smem + C::OFF_DO + st * C::TILE + a * C::BOX, &tm_do, &sh.qdo_full[st], a * C::ATOM, q_row, bh);
          }
          bulk_load(stat + st * 256, lse2_h + q_row, 512, &sh.qdo_full[st]);
          bulk_load(stat + st * 256 + 128, D_h + q_row, 512, &sh.qdo_full[st]);
          if (st == 0) q_last0 = static_cast<int>(ph);
          else if (st == 1) q_last1 = static_cast<int>(ph);
          else q_last2 = static_cast<int>(ph);
        }
      }
      // Let every copy this thread started land before shared memory is released.
      if (kv_last0 >= 0) drain_wait_b(&sh.kv_full[0], static_cast<uint32_t>(kv_last0), wd);
      if (kv_last1 >= 0) drain_wait_b(&sh.kv_full[1], static_cast<uint32_t>(kv_last1), wd);
      if (q_last0 >= 0) drain_wait_b(&sh.qdo_full[0], static_cast<uint32_t>(q_last0), wd);
      if (q_last1 >= 0) drain_wait_b(&sh.qdo_full[1], static_cast<uint32_t>(q_last1), wd);
      if (q_last2 >= 0) drain_wait_b(&sh.qdo_full[2], static_cast<uint32_t>(q_last2), wd);
    }
  } else if (warp == 13 || warp == 14) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads feed the tensor pipe, one per chain of products:
    //   A (warp 13): S^T(t) and dV += P^T(t) dO(t)       (the P path)
    //   B (warp 14): dP^T(t), dQ(t) = dS K, dK += dS^T Q  (the dS path)
    // so that neither chain waits behind the other's barriers: A issues dV(t)
    // and S^T(t+1) as soon as P(t) is in TMEM, while B waits for dS(t) and, at
    // d = 128, for the dQ tile's columns before dP^T(t+1). The two chains use
    // disjoint TMEM columns (S^T | dV for A, dP^T | dK | dQ for B) and share
    // only operands in shared memory, whose stages are released when both
    // threads' products have read them (barriers with two arrivals).
    const bool is_a = (warp == 13);
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
        const int a = k / (C::ATOM / 16), w = k % (C::ATOM / 16);
        const uint64_t da = smem_desc(a_base + a * C::BOX + w * 32, 16, C::SBO, C::SWZ);
        const uint64_t db = smem_desc(b_base + a * C::BOX + w * 32, 16, C::SBO, C::SWZ);
        mma_ss(d_tmem, da, db, idesc, k > 0 ? 1u : 0u);
      }
    };
    // B operand: a [128 rows][D] tile read MN-major, K = 16 rows per step.
    auto b_mn = [&](uint32_t base, int k) {
      return smem_desc(base + k * 16 * C::ATOM * 2, C::BOX, C::SBO, C::SWZ);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, guarded_wait(bar, parity, abort_flag, wd, site));
    };
    bool ok = true;
    int g = 0, li = 0;
    for (int it = blockIdx.x; ok && it < p.num_items; it += gridDim.x, ++li) {
      int bh, kb, i_start, T, rot;
      item_of(it, bh, kb, i_start, T, rot);
      const int set = li % C::KV_SETS, use = li / C::KV_SETS;
      const uint32_t sK = smem_u32(smem + C::OFF_K + set * C::TILE);
      const uint32_t sV = smem_u32(smem + C::OFF_V + set * C::TILE);
      if (!(ok = wait_all(&sh.kv_full[set], use & 1, kSiteBwdLoad))) break;
      // acc_free is waited once per item, in order: before the item's first dV
      // (A) or dK (B) product, or here for an item without query tiles
      if (T == 0 && li >= 1 && !(ok = wait_all(&sh.acc_free, (li - 1) & 1, kSiteBwdFinal))) break;
      if (T > 0) {
        if (!(ok = wait_all(&sh.qdo_full[g % C::QS], (g / C::QS) & 1, kSiteBwdLoad))) break;
        if (is_a) {
          if (lane == 0) {
            tc_fence_after();
            issue_kmajor(tmem + C::TM_S, sK, sQ + (g % C::QS) * C::TILE, id_s);
            mma_commit(&sh.s_full);
          }
        } else {
          // for d = 128 dP shares its TMEM columns with the previous tile's dQ
          if (C::ALIAS_DQ && g >= 1 && !(ok = wait_all(&sh.dq_empty, (g - 1) & 1, kSiteBwdDQ))) break;
          if (lane == 0) {
            tc_fence_after();
            issue_kmajor(tmem + C::TM_DP, sV, sDO + (g % C::QS) * C::TILE, id_dp);
            mma_commit(&sh.dp_full);
          }
        }
        __syncwarp();
      }
      for (int t = 0; ok && t < T; ++t) {
        const int gt = g + t;
        const int st = gt % C::QS, sn = (gt + 1) % C::QS;  // this tile's stage, the next one's
        const uint32_t q_off = st * C::TILE;
        if (is_a) {
          // dV += P^T dO; P^T (bf16) sits in TMEM columns [0,32) and [64,96) of S^T,
          // one block per compute warpgroup (queries 0..63 and 64..127)
          if (!(ok = wait_all(&sh.p_full, gt & 1, kSiteBwdS))) break;
          // The item's first dV product overwrites the accumulator: the previous
          // item's epilogue must have read dK and dV out of TMEM.
          if (t == 0 && li >= 1 && !(ok = wait_all(&sh.acc_free, (li - 1) & 1, kSiteBwdFinal))) break;
          if (lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tmem + C::TM_DV, tmem + C::TM_S + (k >> 2) * 64 + (k & 3) * 8, b_mn(sDO + q_off, k), id_kv,
                     (t > 0 || k > 0) ? 1u : 0u);
          }
          __syncwarp();
          // next S^T (over this tile's P^T, which dV has read by then in the pipe's order)
          if (t + 1 < T) {
            if (!(ok = wait_all(&sh.qdo_full[sn], ((gt + 1) / C::QS) & 1, kSiteBwdLoad))) break;
            if (lane == 0) {
              issue_kmajor(tmem + C::TM_S, sK, sQ + sn * C::TILE, id_s);
              mma_commit(&sh.s_full);
            }
          }
          if (lane == 0) mma_commit(&sh.qdo_empty[st]);  // this thread's reads of Q(t), dO(t) done
          __syncwarp();
        } else {
          if (!(ok = wait_all(&sh.ds_full, gt & 1, kSiteBwdDS))) break;
          if (!C::ALIAS_DQ && gt >= 1) {
            if (!(ok = wait_all(&sh.dq_empty, (gt - 1) & 1, kSiteBwdDQ))) break;
          }
          // The item's first dK product overwrites the accumulator (see above).
          if (t == 0 && li >= 1 && !(ok = wait_all(&sh.acc_free, (li - 1) & 1, kSiteBwdFinal))) break;
          if (lane == 0) {
            tc_fence_after();
            // dQ = dS K first: A = dS (MN-major: queries contiguous), B = K (MN-major).
            // Its drain out of TMEM gates the next dP^T product at d = 128 (the two
            // share columns), so it goes ahead of dK in the tensor pipe's order.
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t da = smem_desc(sDS + k * 16 * 128, C::DS_REGION, 1024, 2);
              mma_ss(tmem + C::TM_DQ, da, b_mn(sK, k), id_dq, k > 0 ? 1u : 0u);
            }
            mma_commit(&sh.dq_full);
            // dK += dS^T Q : A = dS^T (K-major over queries), B = Q (MN-major)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t da = smem_desc(sDS + (k >> 2) * C::DS_REGION + (k & 3) * 32, 16, 1024, 2);
              mma_ss(tmem + C::TM_DK, da, b_mn(sQ + q_off, k), id_kv, (t > 0 || k > 0) ? 1u : 0u);
            }
            if (C::DQ_IN_DS) mma_commit(&sh.dk_done);   // the dQ staging may now overwrite dS
            else mma_commit(&sh.ds_empty);                // (d = 128: the dQ warpgroup releases it)
            mma_commit(&sh.qdo_empty[st]);  // this thread's reads of Q(t), dO(t) done
          }
          __syncwarp();
          if (t + 1 < T) {
            if (C::ALIAS_DQ) {
              if (!(ok = wait_all(&sh.dq_empty, gt & 1, kSiteBwdDQ))) break;
            }
            if (!(ok = wait_all(&sh.qdo_full[sn], ((gt + 1) / C::QS) & 1, kSiteBwdLoad))) break;
            if (lane == 0) {
              tc_fence_after();
              issue_kmajor(tmem + C::TM_DP, sV, sDO + sn * C::TILE, id_dp);
              mma_commit(&sh.dp_full);
            }
            __syncwarp();
          }
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(&sh.dkv_full);      // this thread's accumulator (dV or dK) is complete
        mma_commit(&sh.kv_empty[set]);  // and its reads of K, V are done
      }
      __syncwarp();
      g += T;
    }
    uint64_t* drain = is_a ? &sh.drain : &sh.drain_b;
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    drain_wait_b(drain, 0, wd);
  } else if (warp >= 15) {
    // idle warp: it only completes the fourth warpgroup for the register split
  } else if (warp < 8) {
    // ------------------------------------------------------------ P, dS, dK/dV epilogue
    // Two warpgroups on the same key rows (TMEM lanes): group h owns query
    // columns [64h, 64h+64) of every tile.
    reg_alloc<C::REG_COMPUTE>();
    const int h = warp >> 2;
    const int col0 = 64 * h;
    const int r = tid & 127;                            // key row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::TM_S + col0;
    const uint32_t t_dp = tmem + lane_base + C::TM_DP + col0;
    // Scale 0 runs with a tiny positive c instead of 0, as in the forward: each
    // visible weight stays exactly 2^(-lse * log2 e), and a score of -inf (a masked
    // query) gives weight 0 (-inf * 0 would be NaN), so the exponential loop
    // needs no per-element mask test.
    const float c = p.c > 0.f ? p.c : 1e-30f;
    uint8_t* ds_row = smem + C::OFF_DS + h * C::DS_REGION + r * 128;
    const int sw = r & 7;
    bool ok = true;
    int g = 0, li = 0;
    for (int it = blockIdx.x; ok && it < p.num_items; it += gridDim.x, ++li) {
      int bh, kb, i_start, T, rot;
      item_of(it, bh, kb, i_start, T, rot);
      const int key = kb * 128 + r;
      const int mb = head_keys(p.kv_len, bh, p.h, p.m);  // real keys of this head
      int qlo, qhi;  // query rows that see this key
      query_range(key, key, p.n, p.causal, wl, wr, qlo, qhi);
      // region h carried the previous item's dV / dK out: its TMA store must
      // have read it before dS (or this item's output) overwrites it
      if (C::STAGE_OUT && li >= 1) {
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.out_free[h], (li - 1) & 1, abort_flag, wd, kSiteBwdFinal));
        if (!ok) break;
      }
      for (int t = 0; t < T; ++t) {
        const int gt = g + t;
        const int st = gt % C::QS;
        const int q_row0 = q_tile(i_start, T, rot, t) * 128;
        // queries [lo, hi) of this tile may attend to this key
        const int lo = max(0, qlo - q_row0);
        const int hi = (key < mb) ? min(128, qhi - q_row0) : 0;
        const bool masked = __any_sync(0xffffffffu, lo > col0 || hi < col0 + 64);
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full, gt & 1, abort_flag, wd, kSiteBwdS) &&
                                         guarded_wait(&sh.qdo_full[st], (gt / C::QS) & 1, abort_flag, wd, kSiteBwdLoad));
        if (!ok) break;
        tc_fence_after();
        const float* nlse2_s = stat + st * 256 + col0;  // -lse * log2(e) per query column
        const float* D_s = stat + st * 256 + 128 + col0;
        // P^T in fp32 pairs for dS below; rounded to bf16 for the dV product
        uint64_t P2[32];
        {
          uint32_t s[2][32];
          tmem_ld32(t_s, s[0]);
          tmem_ld32(t_s + 32, s[1]);
          tmem_ld_wait();
          if (masked) {
            // queries outside [lo, hi) do not see this key: score -inf, weight 0
            // (a separate pass keeps the mask test out of the exponential loop,
            // which measured 9-14 % faster for the long sequences)
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int col = col0 + q * 32 + i;
                if (col < lo || col >= hi) s[q][i] = __float_as_uint(-INFINITY);
              }
          }
          const uint64_t c2 = f2_pack(c, c);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 L = *reinterpret_cast<const float4*>(nlse2_s + q * 32 + i4 * 4);
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int col = i4 * 4 + u * 2;
                const uint64_t x2 = fma2(f2_pack(__uint_as_float(s[q][col]), __uint_as_float(s[q][col + 1])), c2,
                                         u ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y));
                float x0, x1;
                f2_unpack(x2, x0, x1);
                P2[q * 16 + i4 * 2 + u] = f2_pack(ex2f(x0), ex2f(x1));
              }
            }
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
      // The wait is taken for items without query tiles too: it keeps these warps
      // from running more than one item ahead of the MMA warp, so that no
      // barrier is waited on two phases ahead.
      ok = __all_sync(0xffffffffu, guarded_wait(&sh.dkv_full, li & 1, abort_flag, wd, kSiteBwdFinal));
      if (!ok) break;
      tc_fence_after();
      const bool store = key < p.m;
      const size_t off = (static_cast<size_t>(bh) * p.m + (store ? key : 0)) * D;
      uint4* dst = reinterpret_cast<uint4*>((h ? p.dk : p.dv) + off);
      const float mul = h ? p.scale : 1.f;
      uint8_t* region = smem + C::OFF_DS + h * C::DS_REGION;
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
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        if (C::STAGE_OUT) {
          // row r of the tile in the map's swizzled layout: 128-byte rows with
          // the 128-byte swizzle (d = 64), 64-byte rows with the 64-byte one (d = 32)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = q * 4 + u;
            const int pc = (D == 64) ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
            *reinterpret_cast<uint4*>(region + r * (D * 2) + (pc << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        } else if (store) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[q * 4 + u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sh.acc_free);
      if (C::STAGE_OUT) {
        // one thread stores the tile; rows past m are clipped by the map
        fence_proxy_async_smem();
        mbar_arrive(&sh.out_staged[h]);
        if (r == 0) {
          if (guarded_wait(&sh.out_staged[h], li & 1, abort_flag, wd, kSiteBwdFinal)) {
            tma_store_3d(h ? &tm_dk : &tm_dv, region, 0, kb * 128, bh);
            tma_store_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&sh.out_free[h]);
        }
      }
      g += T;
    }
  } else {
    // ------------------------------------------------------------ dQ accumulation (warps 8-11)
    reg_dealloc<C::REG_DQ>();
    const int r = tid - 256;                           // query row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_dq = tmem + lane_base + C::TM_DQ;
    uint8_t* stage = smem + (C::DQ_IN_DS ? C::OFF_DS : C::OFF_DQS);
    uint8_t* stage_row = stage + r * 128;
    const int sw = r & 7;
    int g = 0;
    bool stop = false;
    for (int it = blockIdx.x; !stop && it < p.num_items; it += gridDim.x) {
      int bh, kb, i_start, T, rot;
      item_of(it, bh, kb, i_start, T, rot);
      for (int t = 0; t < T; ++t) {
        const int gt = g + t;
        const int qrow0 = q_tile(i_start, T, rot, t) * 128;
        const bool ok = __all_sync(0xffffffffu, guarded_wait(&sh.dq_full, gt & 1, abort_flag, wd, kSiteBwdDQ));
        // Every warp of the group reaches the barriers. The decision to leave is
        // ORed over the group at a barrier, so all four warps leave together
        // even when another role raises the abort flag meanwhile.
#pragma unroll
        for (int round = 0; round < C::DQ_ROUNDS; ++round) {
          // The round's dQ columns leave TMEM first, and after the last round the
          // columns are released at once (for d = 128 the next dP^T product
          // writes them); only then does the group wait for the staging tile.
          tc_fence_after();
          uint32_t v[C::DQ_BOXES_PER_ROUND][32];
#pragma unroll
          for (int b = 0; b < C::DQ_BOXES_PER_ROUND; ++b)
            tmem_ld32(t_dq + (round * C::DQ_BOXES_PER_ROUND + b) * 32, v[b]);  // 32-column boxes of dQ
          tmem_ld_wait();
          if (round == C::DQ_ROUNDS - 1) {
            tc_fence_before();
            mbar_arrive(&sh.dq_empty);
          }
          // the previous reduce must have read the staging tile; for d = 128 the
          // staging tile is the dS buffer, which the dK product reads until dk_done
          bool staged_ok = ok;
          if (ok && r == 0) {
            if (C::DQ_IN_DS && round == 0)
              staged_ok = guarded_wait(&sh.dk_done, gt & 1, abort_flag, wd, kSiteBwdDQ);
            bulk_wait_read_all();
          }
          if (named_bar_or(1, 128, !staged_ok || *abort_flag != 0)) {
            stop = true;
            break;
          }
#pragma unroll
          for (int b = 0; b < C::DQ_BOXES_PER_ROUND; ++b)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(stage_row + b * C::DQ_BOX + ((ch ^ sw) << 4)) =
                  make_uint4(v[b][4 * ch], v[b][4 * ch + 1], v[b][4 * ch + 2], v[b][4 * ch + 3]);
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (r == 0) {
#pragma unroll
            for (int b = 0; b < C::DQ_BOXES_PER_ROUND; ++b)
              tma_reduce_add_2d(&tm_dq, stage + b * C::DQ_BOX, (round * C::DQ_BOXES_PER_ROUND + b) * 32,
                                bh * p.n_pad + qrow0);
            tma_store_commit();
          }
        }
        if (stop) break;
        if (C::DQ_IN_DS && r == 0) {
          // the dS buffer is free for the next tile once these reduces have read it
          bulk_wait_read_all();
          mbar_arrive(&sh.ds_empty);
        }
      }
      g += T;
    }
    // the reduces read shared memory until they complete
    if (r == 0) tma_store_wait_all();
  }

  // bulk stores issued by this thread must complete before the CTA exits
  if (C::STAGE_OUT && (warp == 0 || warp == 4) && lane == 0) tma_store_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int D, bool WIN>
cudaError_t launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdk, const CUtensorMap& tdv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdPreParams& pre,
                         const BwdParams& p, const BwdPostParams& post, int BH, cudaStream_t stream) {
  using C = Bwd<D>;
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_bwd_kernel<D, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  {
    // setmaxnreg.inc waits until registers are free: the split must fit in the
    // registers the CTA is launched with, or the kernel would never proceed.
    static int regs_per_thread[64] = {0};
    if (regs_per_thread[dev & 63] == 0) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, attn_bwd_kernel<D, WIN>)) != cudaSuccess) return e;
      regs_per_thread[dev & 63] = fa.numRegs;
    }
    const int need = 128 * (2 * C::REG_COMPUTE + C::REG_DQ + C::REG_OTHER);  // four warpgroups
    if (regs_per_thread[dev & 63] * C::THREADS < need) return cudaErrorInvalidConfiguration;
  }
  {
    constexpr int RPB = 256 / (D / 8);
    const long long rows = static_cast<long long>(pre.BH) * pre.n_pad;
    const unsigned blocks = static_cast<unsigned>((rows + RPB - 1) / RPB);
    prof_begin(kKindBwdPre, stream);
    attn_bwd_pre_kernel<D><<<blocks, 256, 0, stream>>>(pre);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_end(kKindBwdPre, stream);
  }
  {
    // persistent: one CTA per SM (at most one per work item) loops over items
    static int sm_count[64] = {0};
    if (sm_count[dev & 63] == 0) {
      int c = 0;
      if ((e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      sm_count[dev & 63] = c > 0 ? c : 1;
    }
    BwdParams pp = p;
    pp.BH = BH;
    pp.num_items = BH * p.num_kblocks;
    pp.head_major = p.causal ? 0 : 1;
    const int grid = pp.num_items < sm_count[dev & 63] ? pp.num_items : sm_count[dev & 63];
    prof_begin(kKindBwdMain, stream);
    attn_bwd_kernel<D, WIN><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, pp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_end(kKindBwdMain, stream);
  }
  {
    const long long chunks = static_cast<long long>(post.BH) * post.n * (D / 8);
    const unsigned blocks = static_cast<unsigned>((chunks + 255) / 256);
    prof_begin(kKindBwdPost, stream);
    attn_bwd_post_kernel<D><<<blocks, 256, 0, stream>>>(post);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_end(kKindBwdPost, stream);
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdk, const CUtensorMap& tdv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdPreParams& pre,
                       const BwdParams& p, const BwdPostParams& post, int BH, cudaStream_t stream) {
  const bool win = p.wl >= 0 || p.wr >= 0;
#define ATTN_BWD_CFG(D_)                                                                   \
  (win ? launch_bwd_d<D_, true>(tq, tk, tv, tdk, tdv, tdo, tdq, pre, p, post, BH, stream) \
       : launch_bwd_d<D_, false>(tq, tk, tv, tdk, tdv, tdo, tdq, pre, p, post, BH, stream))
  switch (d) {
    case 32: return ATTN_BWD_CFG(32);
    case 64: return ATTN_BWD_CFG(64);
    case 128: return ATTN_BWD_CFG(128);
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_BWD_CFG
}

}  // namespace attn
