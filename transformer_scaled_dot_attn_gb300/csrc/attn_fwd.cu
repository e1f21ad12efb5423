// Forward kernel: O = softmax(Q K^T * scale) V for every (b, h) head, plus lse.
//
// "Attention Is All You Need", §3.2.1 eq. (1) and Figure 2 (MatMul, Scale,
// Mask (opt.), SoftMax, MatMul), with the decoder mask of §3.2.3. The paper
// runs eq. (1) as plain matrix multiplies on P100s; here both products run on
// the tcgen05 tensor cores and the softmax is streamed over key tiles with a
// running maximum, so the n x m weight matrix never leaves the SM.
//
// One CTA owns 256 query rows of one head as two 128-row tiles Q0, Q1 and
// streams 128-key tiles K_j, V_j through a TMA/mbarrier ring:
//   warp 8      TMA producer: Q0, Q1 once, then K_j and V_j per stage.
//   warp 9      MMA issuer (one lane): S_g = Q_g K_j^T into TMEM, then
//               O_g += P_g V_j with P_g read from TMEM (aliasing S_g).
//   warps 0-3   softmax for Q0, warps 4-7 for Q1: one thread per row. Each
//               loads its S row from TMEM, takes the row max, computes
//               p = 2^(s*c - m) with c = scale*log2(e), accumulates the row
//               sum, writes bf16 P back into TMEM, rescales its O row when the
//               running max grew by more than 2^8, and finally writes O / l
//               and lse.
// The issue order S0(j+1) after PV0(j) lets each softmax group work on tile
// j+1 while the tensor cores run the other group's products; a commit that
// signals S_g(j) also proves PV_g(j-1) finished, so the O rescale needs no
// extra wait. With the causal mask only the key tiles at or below the
// diagonal are loaded and multiplied.
//
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr float kLn2 = 0.69314718055994530942f;
// A stale running max is kept while new scores exceed it by at most 8 in
// log2 units (p <= 256), so most tiles skip the O rescale. Exact after the
// final division by the row sum.
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Fwd {
  static constexpr int STAGES = (D >= 128) ? 2 : 3;
  static constexpr int ATOM = (D >= 64) ? 64 : D;       // bf16 elements per swizzle row
  static constexpr int NATOM = D / ATOM;                 // TMA boxes per 128-row tile
  static constexpr uint32_t SWZ = (D >= 64) ? 2u : 4u;   // descriptor code: 128B / 64B swizzle
  static constexpr uint32_t SBO = 8u * ATOM * 2u;        // bytes between 8-row groups
  static constexpr uint32_t TILE = 128u * D * 2u;        // one 128-row bf16 tile
  static constexpr uint32_t BOX = 128u * ATOM * 2u;      // one TMA box
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
  static constexpr uint32_t SMEM = OFF_V + STAGES * TILE + 1024;  // + alignment slack
  static constexpr int THREADS = 320;
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D;
};

struct FwdShared {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Key tiles needed by query rows [r_lo, r_hi] (r_hi clipped to n-1 by the caller).
__device__ __forceinline__ int key_tiles(int r_hi, int m, int causal) {
  const int kv_hi = causal ? min(r_hi, m - 1) : (m - 1);
  return kv_hi / 128 + 1;
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

template <int D>
__global__ void __launch_bounds__(320, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Fwd<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) FwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int qb = p.causal ? (p.num_qblocks - 1 - static_cast<int>(blockIdx.y)) : blockIdx.y;
  const int q0 = qb * 256;
  volatile int* abort_flag = &sh.abort_flag;
  const Watchdog wd = p.wd;

  const int n0 = key_tiles(min(q0 + 127, p.n - 1), p.m, p.causal);
  const int n1 = (q0 + 128 < p.n) ? key_tiles(min(q0 + 255, p.n - 1), p.m, p.causal) : 0;
  const int nt = max(n0, n1);

  if (tid == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&sh.s_full[g], 1);
      mbar_init(&sh.p_full[g], 128);
      mbar_init(&sh.o_full[g], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc<512>(&sh.tmem_base);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_last[4] = {-1, -1, -1, -1}, v_last[4] = {-1, -1, -1, -1};
      const int nq = (n1 > 0) ? 2 : 1;
      mbar_arrive_expect_tx(&sh.q_full, nq * C::TILE);
      for (int t = 0; t < nq; ++t)
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_Q + t * C::TILE + a * C::BOX, &tm_q, &sh.q_full, a * C::ATOM,
                      q0 + t * 128, bh);
      for (int j = 0; j < nt; ++j) {
        const int st = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        if (j >= C::STAGES && !guarded_wait(&sh.k_empty[st], ph ^ 1, abort_flag, wd, kSiteKEmpty)) break;
        mbar_arrive_expect_tx(&sh.k_full[st], C::TILE);
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_K + st * C::TILE + a * C::BOX, &tm_k, &sh.k_full[st],
                      a * C::ATOM, j * 128, bh);
        k_last[st] = static_cast<int>(ph);
        if (j >= C::STAGES && !guarded_wait(&sh.v_empty[st], ph ^ 1, abort_flag, wd, kSiteVEmpty)) break;
        if (p.inject == 1 && j == 0) continue;  // test hook: this value tile never arrives
        mbar_arrive_expect_tx(&sh.v_full[st], C::TILE);
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(smem + C::OFF_V + st * C::TILE + a * C::BOX, &tm_v, &sh.v_full[st],
                      a * C::ATOM, j * 128, bh);
        v_last[st] = static_cast<int>(ph);
      }
      // Let every copy this thread started land before shared memory is released.
      drain_wait(&sh.q_full, 0, wd);
      for (int s = 0; s < C::STAGES; ++s) {
        if (k_last[s] >= 0) drain_wait(&sh.k_full[s], static_cast<uint32_t>(k_last[s]), wd);
        if (v_last[s] >= 0) drain_wait(&sh.v_full[s], static_cast<uint32_t>(v_last[s]), wd);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false) | (p.neg ? (1u << 13) : 0u);
    const uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    auto issue_s = [&](int g, int st) {
      const uint32_t d_tmem = tmem + (g ? C::TM_S1 : C::TM_S0);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const int a = k / (C::ATOM / 16), w = k % (C::ATOM / 16);
        const uint64_t da = smem_desc(sQ + g * C::TILE + a * C::BOX + w * 32, 16, C::SBO, C::SWZ);
        const uint64_t db = smem_desc(sK + st * C::TILE + a * C::BOX + w * 32, 16, C::SBO, C::SWZ);
        mma_ss(d_tmem, da, db, idesc_s, k > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int g, int st, bool acc) {
      const uint32_t d_tmem = tmem + (g ? C::TM_O1 : C::TM_O0);
      const uint32_t a_tmem = tmem + (g ? C::TM_S1 : C::TM_S0);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t db = smem_desc(sV + st * C::TILE + k * 16 * C::ATOM * 2, C::BOX, C::SBO, C::SWZ);
        mma_ts(d_tmem, a_tmem + k * 8, db, idesc_o, (acc || k > 0) ? 1u : 0u);
      }
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, guarded_wait(bar, parity, abort_flag, wd, site));
    };
    bool ok = wait_all(&sh.q_full, 0, kSiteQFull);
    if (ok && nt > 0) {
      ok = wait_all(&sh.k_full[0], 0, kSiteKFull);
      if (ok && lane == 0) {
        tc_fence_after();
        if (n0 > 0) { issue_s(0, 0); mma_commit(&sh.s_full[0]); }
        if (n1 > 0) { issue_s(1, 0); mma_commit(&sh.s_full[1]); }
        mma_commit(&sh.k_empty[0]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % C::STAGES;
      const uint32_t ph = (j / C::STAGES) & 1;
      const int jn = j + 1, stn = jn % C::STAGES;
      if (!(ok = wait_all(&sh.v_full[st], ph, kSiteVFull))) break;
      if (j < n0) {
        if (!(ok = wait_all(&sh.p_full[0], j & 1, kSitePFull))) break;
        if (lane == 0) {
          tc_fence_after();
          issue_pv(0, st, j > 0);
          if (j == n0 - 1) mma_commit(&sh.o_full[0]);
        }
        __syncwarp();
      }
      if (jn < nt) {
        if (!(ok = wait_all(&sh.k_full[stn], (jn / C::STAGES) & 1, kSiteKFull))) break;
        if (jn < n0 && lane == 0) {
          issue_s(0, stn);
          mma_commit(&sh.s_full[0]);
        }
        __syncwarp();
      }
      if (j < n1) {
        if (!(ok = wait_all(&sh.p_full[1], j & 1, kSitePFull))) break;
        if (lane == 0) {
          tc_fence_after();
          issue_pv(1, st, j > 0);
          if (j == n1 - 1) mma_commit(&sh.o_full[1]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        mma_commit(&sh.v_empty[st]);
        if (jn < nt) {
          if (jn < n1) {
            issue_s(1, stn);
            mma_commit(&sh.s_full[1]);
          }
          mma_commit(&sh.k_empty[stn]);
        }
      }
      __syncwarp();
    }
    // Every MMA this warp issued must finish before TMEM is released.
    if (lane == 0) mma_commit(&sh.drain);
    __syncwarp();
    drain_wait(&sh.drain, 0, wd);
  } else {
    // ------------------------------------------------------------ softmax groups
    const int g = warp >> 2;
    const int r = tid & 127;
    const int row = q0 + g * 128 + r;
    const int ntile = g ? n1 : n0;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + (g ? C::TM_S1 : C::TM_S0);
    const uint32_t t_o = tmem + lane_base + (g ? C::TM_O1 : C::TM_O0);
    const int lim = p.causal ? min(row + 1, p.m) : p.m;  // keys [0, lim) are visible
    const float c = p.c;
    float m_used = 0.f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      ok = __all_sync(0xffffffffu, guarded_wait(&sh.s_full[g], j & 1, abort_flag, wd, kSiteSFull));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(t_s + q * 32, s[q]);
      tmem_ld_wait();
      const int rem = lim - j * 128;  // visible keys of this row inside the tile
      const bool masked = __any_sync(0xffffffffu, rem < 128);
      if (masked) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i >= rem) s[q][i] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(s[0][i]);
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (q > 0 || i >= 8) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(s[q][i]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = mx * c;
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m_used = m_new;
      } else if (m_new > m_used + kRescaleThreshold) {
        alpha = ex2(m_used - m_new);
        m_used = m_new;
        rescale = true;
      }
      const float neg_m = -m_used;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0 = fmaf(__uint_as_float(s[q][2 * i]), c, neg_m);
          float x1 = fmaf(__uint_as_float(s[q][2 * i + 1]), c, neg_m);
          if (masked) {
            if (q * 32 + 2 * i >= rem) x0 = -INFINITY;
            if (q * 32 + 2 * i + 1 >= rem) x1 = -INFINITY;
          }
          const float p0 = ex2(x0), p1 = ex2(x1);
          ls[i & 3] += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + q * 16, pk);
      }
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      tmem_st_wait();
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(t_o + q * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(t_o + q * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&sh.p_full[g]);
    }
    if (ok && ntile > 0) {
      ok = __all_sync(0xffffffffu, guarded_wait(&sh.o_full[g], 0, abort_flag, wd, kSiteOFull));
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const bool store = row < p.n;
        uint4* orow = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.n + (store ? row : 0)) * D);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(t_o + q * 32, o);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (store) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[q * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        if (store && p.lse != nullptr)
          p.lse[static_cast<size_t>(bh) * p.n + row] = (m_used + log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int D>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, int BH, cudaStream_t stream) {
  using C = Fwd<D>;
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>(p.num_qblocks));
  prof_begin(kKindFwd, stream);
  attn_fwd_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  prof_end(kKindFwd, stream);
  return e;
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int BH, cudaStream_t stream) {
  switch (d) {
    case 32: return launch_fwd_d<32>(tq, tk, tv, p, BH, stream);
    case 64: return launch_fwd_d<64>(tq, tk, tv, p, BH, stream);
    case 128: return launch_fwd_d<128>(tq, tk, tv, p, BH, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
